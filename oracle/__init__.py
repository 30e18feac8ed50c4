"""Oracle: the plain CPU definition of the Laya encoder forward pass.

TEST INFRASTRUCTURE ONLY.  This package is the checker the CUDA library is
compared against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
library under ``transformer_encoder_bf16_gb300`` never does, and this package
never imports the library.  The arithmetic lives in ``laya_oracle.c`` (plain C,
fp32 with BF16 storage points, built with ``-ffp-contract=off``); this module
only compiles it and marshals numpy arrays through ctypes.

Inputs are BF16 bit patterns held in ``numpy.uint16`` arrays; outputs are
fp32 arrays whose values are BF16-representable (or raw fp32 sums for
``linear_f32``).  Which passage of the pages each step follows is written
beside each function in ``laya_oracle.c``.  Parity status: each step is pinned
by ``tests/test_oracle_*.py``; the full-stack values at the real sizes have no
published numbers to pin them to ("parity unpinned" beyond the pinned steps and
the stack invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "laya_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liblaya_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile laya_oracle.c into liblaya_oracle.so (gcc, OpenMP if present)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


class OrcConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "heads", "head_dim", "intermediate", "vocab",
        "n_encoder_layers", "n_decision_layers", "global_every",
        "local_half_window")] + [
        ("theta_global", ctypes.c_float), ("theta_local", ctypes.c_float),
        ("ln_eps", ctypes.c_float)] + [(n, ctypes.c_int32) for n in (
            "max_seq", "rope_table_bf16", "first_attn_norm_identity",
            "final_norm", "accum_f64", "out_fp32")]


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.orc_abi.restype = _I
            L.orc_set_threads.argtypes = [_I]
            L.orc_set_threads.restype = _I
            L.orc_bf16_round.argtypes = [_F]
            L.orc_bf16_round.restype = _F
            L.orc_gelu.argtypes = [_F]
            L.orc_gelu.restype = _F
            L.orc_rope_table.argtypes = [ctypes.c_double, _I, _I, _I, _P, _P]
            L.orc_rope_vec.argtypes = [_P, _P, _P, _I]
            L.orc_layernorm_row.argtypes = [_P, _P, _I, _F, _P]
            L.orc_step_layernorm.argtypes = [_P, _P, _I, _I, _F, _P]
            L.orc_step_linear_f32.argtypes = [_P, _I, _I, _P, _I, _I, _P]
            L.orc_step_linear.argtypes = [_P, _I, _I, _P, _I, _I, _P, _P]
            L.orc_step_rope.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P]
            L.orc_step_attention.argtypes = [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P]
            L.orc_step_embed_layernorm.argtypes = [_P, _P, _P, _I, _I, _F, _P]
            L.orc_forward.argtypes = [ctypes.POINTER(OrcConfig), _P, _P, _P, _P,
                                      _P, _P, _I, _I, _P, _I, _P]
            L.orc_forward.restype = _I
            L.orc_layer.argtypes = [ctypes.POINTER(OrcConfig), _I, _P, _P, _P, _I, _I, _P, _P]
            L.orc_layer.restype = _I
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def set_threads(n: int) -> int:
    """Set the OpenMP thread count for later calls; returns the count in use."""
    return lib().orc_set_threads(int(n))


def bf16_round(x: float) -> float:
    return lib().orc_bf16_round(float(x))


def gelu(z: float) -> float:
    return lib().orc_gelu(float(z))


def make_config(model: dict, accum_f64: bool = False, out_fp32: bool = False) -> OrcConfig:
    c = OrcConfig()
    for name, _ in OrcConfig._fields_:
        if name in ("accum_f64", "out_fp32"):
            continue
        setattr(c, name, model[name])
    c.accum_f64 = 1 if accum_f64 else 0
    c.out_fp32 = 1 if out_fp32 else 0
    return c


def rope_table(theta: float, max_seq: int, half: int, bf16: bool = True):
    """fp32 cos/sin tables [max_seq, half]."""
    c = np.zeros((max_seq, half), np.float32)
    s = np.zeros((max_seq, half), np.float32)
    lib().orc_rope_table(float(theta), max_seq, half, 1 if bf16 else 0, _ptr(c), _ptr(s))
    return c, s


def rope_vec(v, c, s):
    """Rotate one head vector (fp32 values, length 2*half) with table rows c, s."""
    v = _f32(v).copy()
    c, s = _f32(c), _f32(s)
    lib().orc_rope_vec(_ptr(v), _ptr(c), _ptr(s), len(c))
    return v


def layernorm_row(x, gamma, eps):
    x, gamma = _f32(x), _f32(gamma)
    y = np.zeros_like(x)
    lib().orc_layernorm_row(_ptr(x), _ptr(gamma), x.shape[-1], float(eps), _ptr(y))
    return y


def layernorm(x_bits, gamma_bits, eps):
    x_bits, gamma_bits = _u16(x_bits), _u16(gamma_bits)
    rows, n = x_bits.shape
    y = np.zeros_like(x_bits)
    lib().orc_step_layernorm(_ptr(x_bits), _ptr(gamma_bits), rows, n, float(eps), _ptr(y))
    return y


def linear_f32(x_bits, w_bits, f64=False):
    x_bits, w_bits = _u16(x_bits), _u16(w_bits)
    rows, k = x_bits.shape
    out = w_bits.shape[0]
    y = np.zeros((rows, out), np.float32)
    lib().orc_step_linear_f32(_ptr(x_bits), rows, k, _ptr(w_bits), out, 1 if f64 else 0, _ptr(y))
    return y


LINEAR_PLAIN, LINEAR_RESIDUAL, LINEAR_GEGLU = 0, 1, 2


def linear(x_bits, w_bits, kind=LINEAR_PLAIN, residual_bits=None):
    x_bits, w_bits = _u16(x_bits), _u16(w_bits)
    rows, k = x_bits.shape
    out = w_bits.shape[0]
    ncol = out // 2 if kind == LINEAR_GEGLU else out
    y = np.zeros((rows, ncol), np.uint16)
    r = _u16(residual_bits) if residual_bits is not None else None
    lib().orc_step_linear(_ptr(x_bits), rows, k, _ptr(w_bits), out, kind, _ptr(r), _ptr(y))
    return y


def rope(qkv_bits, B, S, heads, head_dim, cos_t, sin_t):
    """RoPE of the q and k slices of a packed [B*S, 3H] projection (copy)."""
    q = _u16(qkv_bits).copy()
    H = heads * head_dim
    lib().orc_step_rope(_ptr(q), B, S, H, heads, head_dim, _ptr(_f32(cos_t)), _ptr(_f32(sin_t)))
    return q


def attention(qkv_bits, lengths, B, S, heads, head_dim, global_, half_window):
    qkv_bits = _u16(qkv_bits)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    H = heads * head_dim
    ctx = np.zeros((B * S, H), np.uint16)
    lib().orc_step_attention(_ptr(qkv_bits), _ptr(lengths), B, S, H, heads, head_dim,
                             1 if global_ else 0, half_window, _ptr(ctx))
    return ctx


def embed_layernorm(emb_bits, gamma_bits, ids, eps):
    emb_bits, gamma_bits = _u16(emb_bits), _u16(gamma_bits)
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(-1)
    H = emb_bits.shape[1]
    x = np.zeros((ids.size, H), np.uint16)
    lib().orc_step_embed_layernorm(_ptr(emb_bits), _ptr(gamma_bits), _ptr(ids), ids.size, H,
                                   float(eps), _ptr(x))
    return x


LAYER_KEYS = ("attn_norm", "wqkv", "wo", "mlp_norm", "wup", "wdown")


def forward(model: dict, weights: dict, ids, lengths, accum_f64=False,
            capture_layer=-1, out_fp32=False):
    """Full stack.  ids [B, S] int32, lengths [B] int32.  Returns fp32 [B, S, H]
    (BF16 values; with out_fp32, the last residual sum before its BF16
    rounding), or (out, captured) when capture_layer >= 0."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    B, S = ids.shape
    H = model["hidden"]
    cfg = make_config(model, accum_f64, out_fp32)
    keep = []
    ptrs = []
    for layer in weights["layers"]:
        for key in LAYER_KEYS:
            a = layer.get(key)
            if a is None:
                ptrs.append(None)
            else:
                a = _u16(a)
                keep.append(a)
                ptrs.append(a.ctypes.data)
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    emb = _u16(weights["tok_emb"])
    en = _u16(weights["emb_norm"])
    fn = _u16(weights["final_norm"])
    out = np.zeros((B, S, H), np.float32)
    cap = np.zeros((B, S, H), np.float32) if capture_layer >= 0 else None
    rc = lib().orc_forward(ctypes.byref(cfg), _ptr(emb), _ptr(en), _ptr(fn),
                           ctypes.cast(arr, ctypes.c_void_p), _ptr(ids), _ptr(lengths),
                           B, S, _ptr(out), int(capture_layer), _ptr(cap))
    if rc != 0:
        raise ValueError(f"oracle forward rejected its arguments (rc={rc})")
    return (out, cap) if capture_layer >= 0 else out


def layer(model: dict, weights: dict, l: int, x_in, lengths, accum_f64=False, out_fp32=False):
    """Layer l alone (0-based over the encoder, then the decision layers) on
    the residual stream x_in [B, S, H] (fp32 holding BF16 values); the final
    LayerNorm is applied first when l is the first decision layer.  Returns
    fp32 [B, S, H].  Chaining it from the embedding output reproduces
    forward() bit for bit."""
    x_in = _f32(x_in)
    lengths = np.ascontiguousarray(lengths, dtype=np.int32)
    B, S, H = x_in.shape
    cfg = make_config(model, accum_f64, out_fp32)
    if not 0 <= l < len(weights["layers"]):
        raise ValueError(f"oracle layer: no layer {l}")
    lw = weights["layers"][l]
    keep = [None if lw.get(k) is None else _u16(lw[k]) for k in LAYER_KEYS]
    arr = (ctypes.c_void_p * 6)(*[None if a is None else a.ctypes.data for a in keep])
    fn = _u16(weights["final_norm"]) if weights.get("final_norm") is not None else None
    out = np.zeros((B, S, H), np.float32)
    rc = lib().orc_layer(ctypes.byref(cfg), int(l), ctypes.cast(arr, ctypes.c_void_p), _ptr(fn),
                         _ptr(lengths), B, S, _ptr(x_in), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle layer rejected its arguments (rc={rc})")
    return out
