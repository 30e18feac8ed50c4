"""Laya BF16 encoder forward pass on one GB300 (sm_103a): Python binding.

A thin ctypes layer over ``lib/liblaya_enc.so`` (the C ABI declared in
``include/laya_enc.h`` and ``include/laya_ops.h``).  Functions keep the C
names without their prefix and only marshal arguments: device tensors are
passed as raw pointers, streams as ``cudaStream_t`` handles.  PyTorch is used
by callers for device memory and streams; every step of the forward pass runs
in the library's CUDA kernels.  There is no CPU fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import synth  # noqa: F401  (seeded inputs; no arithmetic of the method)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "liblaya_enc.so")

OK, E_INVAL, E_NOMEM, E_CUDA, E_POISONED, E_UNSUPPORTED, E_DEVICE = 0, -1, -2, -3, -4, -5, -6
ERROR_NAMES = {E_INVAL: "LAYA_E_INVAL", E_NOMEM: "LAYA_E_NOMEM", E_CUDA: "LAYA_E_CUDA",
               E_POISONED: "LAYA_E_POISONED", E_UNSUPPORTED: "LAYA_E_UNSUPPORTED",
               E_DEVICE: "LAYA_E_DEVICE"}
KIND_PLAIN, KIND_RESIDUAL, KIND_GEGLU = 0, 1, 2
# GeGLU from interleaved 128-row weight tiles (64 rows of each half): the
# KIND_GEGLU result bit for bit, same weight layout; N % 64 == 0, unsplit
KIND_GEGLU_IL = 3
PROFILE_CLASSES = ("embed_norm", "norm", "qkv", "rope", "attention", "out_proj", "up_geglu",
                   "down", "output")


class LayaError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "heads", "head_dim", "intermediate", "vocab", "n_encoder_layers",
        "n_decision_layers", "global_every", "local_half_window")] + [
        ("theta_global", ctypes.c_float), ("theta_local", ctypes.c_float),
        ("ln_eps", ctypes.c_float)] + [(n, ctypes.c_int32) for n in (
            "max_batch", "max_seq", "rope_table_bf16", "first_attn_norm_identity",
            "final_norm", "out_fp32")]

    @classmethod
    def from_model(cls, model: dict) -> "Config":
        """Every field from the model dict; out_fp32 defaults to 0 (BF16 output)."""
        c = cls()
        for name, _ in cls._fields_:
            setattr(c, name, model.get(name, 0) if name == "out_fp32" else model[name])
        return c


class CacheStats(ctypes.Structure):
    _fields_ = [("shapes", ctypes.c_int32), ("max_shapes", ctypes.c_int32)] + [
        (n, ctypes.c_uint64) for n in ("bytes", "max_bytes", "created", "evicted", "captures",
                                       "retargets")] + [
        ("setup_ms", ctypes.c_double), ("capture_ms", ctypes.c_double)]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wqkv", "wo", "mlp_norm", "wup", "wdown")]


class Weights(ctypes.Structure):
    _fields_ = [("tok_emb", ctypes.c_void_p), ("emb_norm", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("n_layers", ctypes.c_int32),
                ("layers", ctypes.POINTER(LayerWeights))]


_lib = None
_P, _I, _F, _D, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_size_t

# name -> (argtypes, restype)
_SIGNATURES = {
    "laya_enc_abi_version": ([], _I),
    "laya_enc_validate_config": ([ctypes.POINTER(Config)], _I),
    "laya_enc_create": ([ctypes.POINTER(Config), ctypes.POINTER(Weights), ctypes.POINTER(_P)], _I),
    "laya_enc_run": ([_P, _P, _P, _I, _I, _P, _P], _I),
    "laya_enc_run_device": ([_P, _P, _P, _I, _I, _P, _P], _I),
    "laya_enc_check": ([_P, _P], _I),
    "laya_enc_set_graphs": ([_P, _I], _I),
    "laya_enc_debug_fail_next_run": ([_P], _I),
    "laya_enc_debug_capture": ([_P, _P, _P, _I, _I, _P, _P, _P], _I),
    "laya_enc_debug_set_wait_limit_ns": ([_P, ctypes.c_uint64], _I),
    "laya_enc_debug_withhold_next_run": ([_P], _I),
    "laya_enc_get_cache_stats": ([_P, _P], _I),
    "laya_enc_launch_count": ([_P, _I, _I], _I),
    "laya_enc_workspace_bytes": ([_P, _I, _I, ctypes.POINTER(_SZ)], _I),
    "laya_enc_get_plans": ([_P, _I, _I, _P], _I),
    "laya_enc_set_profiling": ([_P, _I], _I),
    "laya_enc_profile_read": ([_P, ctypes.POINTER(_D), ctypes.POINTER(_I), _I], _I),
    "laya_enc_destroy": ([_P], _I),
    "laya_enc_last_error": ([_P], ctypes.c_char_p),
    "laya_op_embed_layernorm": ([_P, _P, _P, _I, _I, _I, _F, _P, _P, _P], _I),
    "laya_op_layernorm": ([_P, _P, _I, _I, _F, _P, _P], _I),
    "laya_op_rope_table": ([_D, _I, _I, _I, _P, _P], _I),
    "laya_op_rope": ([_P, _P, _P, _I, _I, _I, _I, _P], _I),
    "laya_op_attention": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "laya_op_attention_tc": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "laya_op_attention_rows": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "laya_enc_run_markers": ([_P, _P, _P, _I, _I, _P, _I, _P, _P], _I),
    "laya_op_attention_rope": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "laya_op_linear": ([_P, _I, _I, _P, _I, _I, _P, _P, _P, _SZ, _I, _I, _P], _I),
    "laya_op_linear_noalloc": ([_P, _I, _I, _P, _I, _I, _P, _P, _I, _I, _P], _I),
    "laya_op_linear_ex": ([_P, _I, _I, _P, _I, _I, _P, _P, _P, _SZ, _I, _I, _I, _P], _I),
    "laya_op_linear_workspace_size": ([_I, _I, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "laya_op_linear_ln": ([_P, _P, _F, _I, _I, _P, _I, _I, _P, _P, _P, _SZ, _I, _I, _P], _I),
    "laya_op_linear_rope": ([_P, _I, _I, _P, _I, _P, _P, _I, _I, _P, _P, _SZ, _I, _I, _P], _I),
    "laya_op_linear_plan": ([_I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I),
                             ctypes.POINTER(_I)], _I),
}


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m transformer_encoder_bf16_gb300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (argt, rest) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = argt
            fn.restype = rest
        _lib = L
    return _lib


def _check(rc, handle=None):
    if rc != OK:
        msg = lib().laya_enc_last_error(handle).decode() if handle is not None else "see arguments"
        raise LayaError(rc, msg)
    return rc


def _stream_ptr(stream):
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream  # torch.cuda.Stream


def _ptr(t):
    return None if t is None else t.data_ptr()


# ------------------------------------------------------------- full stack ---

def upload_weights(weights: dict, device="cuda"):
    """Copy the uint16 BF16 bit patterns of synth.make_weights to device
    tensors (torch.bfloat16).  Returns a dict of the same shape."""
    import torch

    def up(a):
        if a is None:
            return None
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)

    return {"tok_emb": up(weights["tok_emb"]), "emb_norm": up(weights["emb_norm"]),
            "final_norm": up(weights["final_norm"]),
            "layers": [{k: up(v) for k, v in layer.items()} for layer in weights["layers"]]}


def check_device_inputs(ids_dev, lengths_dev):
    """The C ABI reads B * S and B int32 values through bare pointers: check
    the tensors' element type, layout and agreement here."""
    import torch
    ok = (ids_dev.dtype == torch.int32 and lengths_dev.dtype == torch.int32 and
          ids_dev.dim() == 2 and lengths_dev.dim() == 1 and ids_dev.is_contiguous() and
          lengths_dev.is_contiguous() and lengths_dev.shape[0] == ids_dev.shape[0] and
          ids_dev.is_cuda and lengths_dev.is_cuda)
    if not ok:
        raise LayaError(E_INVAL, "token ids must be a contiguous int32 [B, S] and lengths a "
                                 "contiguous int32 [B] tensor on the device")


class Encoder:
    """Owns a laya_enc_handle over device weights (kept referenced here)."""

    def __init__(self, model: dict, dev_weights: dict):
        self.model = model
        self._weights = dev_weights
        self._cfg = Config.from_model(model)
        layers = dev_weights["layers"]
        arr = (LayerWeights * len(layers))()
        for i, lw in enumerate(layers):
            for k in ("attn_norm", "wqkv", "wo", "mlp_norm", "wup", "wdown"):
                setattr(arr[i], k, _ptr(lw[k]))
        self._layers = arr
        w = Weights(_ptr(dev_weights["tok_emb"]), _ptr(dev_weights["emb_norm"]),
                    _ptr(dev_weights["final_norm"]), len(layers),
                    ctypes.cast(arr, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        rc = lib().laya_enc_create(ctypes.byref(self._cfg), ctypes.byref(w), ctypes.byref(h))
        if rc != OK:
            raise LayaError(rc, lib().laya_enc_last_error(None).decode())
        self.handle = h

    def run(self, ids: np.ndarray, lengths: np.ndarray, out, stream=None):
        """ids int32 [B, S] and lengths int32 [B] in HOST memory; out a device
        tensor [B, S, hidden], bfloat16 (float32 when the model sets out_fp32)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        B, S = ids.shape
        self._check_out(out, B, S)
        _check(lib().laya_enc_run(self.handle, ids.ctypes.data, lengths.ctypes.data, B, S,
                                  _ptr(out), _stream_ptr(stream)), self.handle)

    def run_markers(self, ids: np.ndarray, lengths: np.ndarray, marker_pos: np.ndarray, out,
                    stream=None):
        """The forward with the last layer at marker rows only.  marker_pos int32
        [B, kmax] in HOST memory (a position in the row, or -1 for an empty
        slot); out a device tensor [B * kmax, hidden] (bfloat16, float32 when
        the model sets out_fp32)."""
        import torch
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        marker_pos = np.ascontiguousarray(marker_pos, dtype=np.int32)
        B, S = ids.shape
        if marker_pos.ndim != 2 or marker_pos.shape[0] != B:
            raise LayaError(E_INVAL, "marker_pos must be an int32 [B, kmax] array")
        kmax = marker_pos.shape[1]
        want = torch.float32 if self._cfg.out_fp32 else torch.bfloat16
        if out.dtype != want or not out.is_contiguous() or out.numel() < B * kmax * self._cfg.hidden:
            raise LayaError(E_INVAL, f"out must be a contiguous {want} tensor of at least "
                                     f"{B * kmax}x{self._cfg.hidden} elements")
        _check(lib().laya_enc_run_markers(self.handle, ids.ctypes.data, lengths.ctypes.data, B, S,
                                          marker_pos.ctypes.data, kmax, _ptr(out),
                                          _stream_ptr(stream)), self.handle)

    def run_device(self, ids_dev, lengths_dev, out, stream=None):
        """ids_dev int32 [B, S] and lengths_dev int32 [B] device tensors."""
        check_device_inputs(ids_dev, lengths_dev)
        B, S = ids_dev.shape
        self._check_out(out, B, S)
        _check(lib().laya_enc_run_device(self.handle, _ptr(ids_dev), _ptr(lengths_dev), B, S,
                                         _ptr(out), _stream_ptr(stream)), self.handle)

    def _check_out(self, out, B, S):
        # the C ABI takes a bare pointer: the element type and size are checked here
        import torch
        want = torch.float32 if self._cfg.out_fp32 else torch.bfloat16
        if out.dtype != want or not out.is_contiguous() or out.numel() < B * S * self._cfg.hidden:
            raise LayaError(E_INVAL, f"out must be a contiguous {want} tensor of at least "
                                     f"{B}x{S}x{self._cfg.hidden} elements")

    def check(self, stream=None):
        return _check(lib().laya_enc_check(self.handle, _stream_ptr(stream)), self.handle)

    def debug_fail_next_run(self):
        """Test hook: the next run fails like a CUDA launch failure (poisons the handle)."""
        _check(lib().laya_enc_debug_fail_next_run(self.handle), self.handle)

    def debug_set_wait_limit_ns(self, ns: int):
        """Bound of the projections' barrier waits (0: the default 2 s)."""
        _check(lib().laya_enc_debug_set_wait_limit_ns(self.handle, int(ns)), self.handle)

    def debug_withhold_next_run(self):
        """Test hook: the next run's first projection withholds one pipeline
        stage, so a bounded wait runs out (LAYA_E_DEVICE at check())."""
        _check(lib().laya_enc_debug_withhold_next_run(self.handle), self.handle)

    def set_graphs(self, enabled: bool):
        _check(lib().laya_enc_set_graphs(self.handle, 1 if enabled else 0), self.handle)

    def debug_capture(self, ids: np.ndarray, lengths: np.ndarray, out, states, stream=None):
        """As run(), eagerly, also writing states [L, B, S, hidden] bfloat16:
        the residual stream entering every layer (padded layout, padding 0)."""
        import torch
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        lengths = np.ascontiguousarray(lengths, dtype=np.int32)
        B, S = ids.shape
        self._check_out(out, B, S)
        L = self.model["n_encoder_layers"] + self.model["n_decision_layers"]
        if (states.dtype != torch.bfloat16 or not states.is_contiguous() or not states.is_cuda
                or states.numel() < L * B * S * self._cfg.hidden):
            raise LayaError(E_INVAL, f"states must be a contiguous bfloat16 device tensor of at "
                                     f"least {L}x{B}x{S}x{self._cfg.hidden} elements")
        _check(lib().laya_enc_debug_capture(self.handle, ids.ctypes.data, lengths.ctypes.data, B, S,
                                            _ptr(out), _ptr(states), _stream_ptr(stream)),
               self.handle)

    def set_profiling(self, enabled: bool):
        _check(lib().laya_enc_set_profiling(self.handle, 1 if enabled else 0), self.handle)

    def profile_read(self) -> dict:
        """{class: (total device ms, launches)} since the last read."""
        n = len(PROFILE_CLASSES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int * n)()
        _check(lib().laya_enc_profile_read(self.handle, ms, cnt, n), self.handle)
        return {PROFILE_CLASSES[i]: (ms[i], cnt[i]) for i in range(n)}

    def cache_stats(self) -> dict:
        """The workspace / graph cache counters (laya_enc_get_cache_stats)."""
        st = CacheStats()
        _check(lib().laya_enc_get_cache_stats(self.handle, ctypes.byref(st)), self.handle)
        return {name: getattr(st, name) for name, _ in CacheStats._fields_}

    def launch_count(self, B, S) -> int:
        return lib().laya_enc_launch_count(self.handle, B, S)

    def plans(self, B, S) -> dict:
        """{projection: (tokens per tile, split-K, pairing, CTAs, kind)} of a shape that has run."""
        out = (ctypes.c_int32 * 20)()
        _check(lib().laya_enc_get_plans(self.handle, B, S, out), self.handle)
        return {n: tuple(out[5 * g: 5 * g + 5])
                for g, n in enumerate(("qkv", "out_proj", "up_geglu", "down"))}

    def workspace_bytes(self, B, S) -> int:
        n = ctypes.c_size_t()
        _check(lib().laya_enc_workspace_bytes(self.handle, B, S, ctypes.byref(n)), self.handle)
        return n.value

    def last_error(self) -> str:
        return lib().laya_enc_last_error(self.handle).decode()

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().laya_enc_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def abi_version() -> int:
    return lib().laya_enc_abi_version()


def validate_config(model: dict) -> int:
    return lib().laya_enc_validate_config(ctypes.byref(Config.from_model(model)))


# ------------------------------------------------------------ single steps ---

def embed_layernorm(emb, gamma, ids_dev, eps, x, err_dev=None, stream=None):
    M = ids_dev.numel()
    V, H = emb.shape
    _check(lib().laya_op_embed_layernorm(_ptr(emb), _ptr(gamma), _ptr(ids_dev), M, H, V, eps,
                                         _ptr(x), _ptr(err_dev), _stream_ptr(stream)))


def layernorm(x, gamma, eps, y, stream=None):
    M, H = x.shape
    _check(lib().laya_op_layernorm(_ptr(x), _ptr(gamma), M, H, eps, _ptr(y), _stream_ptr(stream)))


def rope_table(theta, max_seq, half, bf16=True):
    c = np.zeros((max_seq, half), np.float32)
    s = np.zeros((max_seq, half), np.float32)
    _check(lib().laya_op_rope_table(float(theta), max_seq, half, 1 if bf16 else 0,
                                    c.ctypes.data, s.ctypes.data))
    return c, s


def rope(qkv, cos_dev, sin_dev, B, S, heads, head_dim=64, stream=None):
    _check(lib().laya_op_rope(_ptr(qkv), _ptr(cos_dev), _ptr(sin_dev), B, S, heads, head_dim,
                              _stream_ptr(stream)))


def attention(qkv, lengths_dev, B, S, heads, global_, half_window, ctx, head_dim=64, stream=None):
    _check(lib().laya_op_attention(_ptr(qkv), _ptr(lengths_dev), B, S, heads, head_dim,
                                   1 if global_ else 0, half_window, _ptr(ctx),
                                   _stream_ptr(stream)))


def attention_tc(qkv, lengths_dev, B, S, heads, global_, half_window, ctx, head_dim=64, stream=None):
    """attention() on the tcgen05 kernel (TMEM accumulators, TMA tiles)."""
    _check(lib().laya_op_attention_tc(_ptr(qkv), _ptr(lengths_dev), B, S, heads, head_dim,
                                      1 if global_ else 0, half_window, _ptr(ctx),
                                      _stream_ptr(stream)))


def attention_rows(qkv, lengths_dev, q_tok_dev, q_pos_dev, B, S, kmax, heads, global_,
                   half_window, ctx_rows, head_dim=64, stream=None):
    """Attention from the query slots q_tok_dev / q_pos_dev (int32 [B * kmax]) of each row."""
    _check(lib().laya_op_attention_rows(_ptr(qkv), _ptr(lengths_dev), _ptr(q_tok_dev),
                                        _ptr(q_pos_dev), B, S, kmax, heads, head_dim,
                                        1 if global_ else 0, half_window, _ptr(ctx_rows),
                                        _stream_ptr(stream)))


def attention_rope(qkv, lengths_dev, cos_dev, sin_dev, B, S, heads, global_, half_window, ctx,
                   head_dim=64, stream=None):
    _check(lib().laya_op_attention_rope(_ptr(qkv), _ptr(lengths_dev), _ptr(cos_dev), _ptr(sin_dev),
                                        B, S, heads, head_dim, 1 if global_ else 0, half_window,
                                        _ptr(ctx), _stream_ptr(stream)))


def linear(x, w, y, kind=KIND_PLAIN, residual=None, splits=0, tile_tokens=0, stream=None,
           workspace=None, paired=0):
    """workspace: a device tensor of at least linear_workspace_size() bytes; a
    fresh one is allocated when None (pass one when capturing a graph).
    paired: 0, or the persistent kernel in clusters of two sharing the token
    tile (1) or the weight tiles (2) of every stage, or issuing one two-CTA
    MMA per pair of feature tiles (3) (splits must be 1)."""
    M, K = x.shape
    N = y.shape[1]
    ws = workspace if workspace is not None else _workspace(M, K, N, kind, splits, tile_tokens, y.device)
    _check(lib().laya_op_linear_ex(_ptr(x), M, K, _ptr(w), N, kind, _ptr(residual), _ptr(y),
                                   _ptr(ws), ws.numel() if ws is not None else 0, splits,
                                   tile_tokens, int(paired), _stream_ptr(stream)))


def linear_noalloc(x, w, y, kind=KIND_PLAIN, residual=None, splits=0, tile_tokens=0, stream=None):
    """linear() without a workspace argument: the library's fixed 16 MiB device
    array holds the split-K partials (for callers that cannot allocate)."""
    M, K = x.shape
    N = y.shape[1]
    _check(lib().laya_op_linear_noalloc(_ptr(x), M, K, _ptr(w), N, kind, _ptr(residual), _ptr(y),
                                        splits, tile_tokens, _stream_ptr(stream)))


def linear_workspace_size(M, K, N, kind, splits=0, tile_tokens=0) -> int:
    n = ctypes.c_size_t()
    _check(lib().laya_op_linear_workspace_size(M, K, N, kind, splits, tile_tokens, ctypes.byref(n)))
    return n.value


def _workspace(M, K, N, kind, splits, tile_tokens, device):
    """A device scratch tensor of the size the plan needs (None when it needs none)."""
    import torch
    n = linear_workspace_size(M, K, N, kind, splits, tile_tokens)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device) if n else None


def linear_ln(x_raw, gamma, eps, w, y, kind=KIND_PLAIN, residual=None, splits=0, tile_tokens=0,
              stream=None, workspace=None):
    M, K = x_raw.shape
    N = y.shape[1]
    ws = workspace if workspace is not None else _workspace(M, K, N, kind, splits, tile_tokens, y.device)
    _check(lib().laya_op_linear_ln(_ptr(x_raw), _ptr(gamma), eps, M, K, _ptr(w), N, kind,
                                   _ptr(residual), _ptr(y), _ptr(ws), ws.numel() if ws is not None else 0,
                                   splits, tile_tokens, _stream_ptr(stream)))


def linear_rope(x, w, y, cos_dev, sin_dev, S, rope_cols, splits=0, tile_tokens=0, stream=None,
                workspace=None):
    M, K = x.shape
    N = y.shape[1]
    ws = workspace if workspace is not None else _workspace(M, K, N, KIND_PLAIN, splits, tile_tokens,
                                                             y.device)
    _check(lib().laya_op_linear_rope(_ptr(x), M, K, _ptr(w), N, _ptr(cos_dev), _ptr(sin_dev), S,
                                     rope_cols, _ptr(y), _ptr(ws), ws.numel() if ws is not None else 0,
                                     splits, tile_tokens, _stream_ptr(stream)))


def linear_plan(M, K, N, kind, num_sms):
    nt, sp, ct = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().laya_op_linear_plan(M, K, N, kind, num_sms, ctypes.byref(nt), ctypes.byref(sp),
                                     ctypes.byref(ct)))
    return nt.value, sp.value, ct.value
