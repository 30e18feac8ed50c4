"""Seeded synthetic inputs for the Laya encoder: model shapes, weights, ids.

This module holds no arithmetic of the method.  It only draws random numbers
and rounds them to BF16 bit patterns, so that the CUDA library and the CPU
oracle are fed identical bytes.  There is no checkpoint: weights are
N(0, 0.02) draws, LayerNorm gammas are 1 + N(0, 0.02), token ids are uniform
over the vocabulary, and padded batches draw their row lengths uniformly from
the stated range (right padding, ids of padded slots drawn too).

Shapes follow the pages: a 28-layer encoder plus 2 decision layers
("Run Laya encoder and decision layers on CUDA", section "H800 comparison"),
at most 16 rows of at most 512 tokens ("Laya native CUDA worker", section
"Start and check"), hidden 1024 with 16 heads of 64, GeGLU width 2624 and a
50368-token vocabulary (the sizes of a 421M-parameter encoder, "[Performance]:
Optimize native Rust/CUDA Laya inference #66", section "Recorded baseline and
environment"), plus a reduced 4+1-layer model at hidden 256 for fast checks.
"""
from __future__ import annotations

import numpy as np

# Model shapes.  Keys match the fields of the library's configuration struct.
_COMMON = dict(
    head_dim=64,
    global_every=3,
    local_half_window=64,
    theta_global=160000.0,
    theta_local=10000.0,
    ln_eps=1e-5,
    max_seq=512,
    max_batch=16,
    rope_table_bf16=1,
    first_attn_norm_identity=1,
    final_norm=1,
)

REDUCED = dict(_COMMON, name="reduced-h256", hidden=256, heads=4, intermediate=640,
               vocab=4096, n_encoder_layers=4, n_decision_layers=1)

FULL = dict(_COMMON, name="laya-encoder-28+2", hidden=1024, heads=16, intermediate=2624,
            vocab=50368, n_encoder_layers=28, n_decision_layers=2)

# Workloads: (model, batch, seq, seed, (len_lo, len_hi) or None for full rows).
WORKLOADS = {
    "reduced_1x48": (REDUCED, 1, 48, 0, None),
    "full_1x48": (FULL, 1, 48, 1, None),
    "full_4x64": (FULL, 4, 64, 2, (16, 64)),
    "full_1x464": (FULL, 1, 464, 2, None),
    "full_4x464": (FULL, 4, 464, 3, None),
    "full_16x512": (FULL, 16, 512, 4, (32, 512)),
}


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to BF16 (nearest, ties to even) and return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bits(rng, shape, std, mean=0.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    x *= np.float32(std)
    if mean:
        x += np.float32(mean)
    return f32_to_bf16_bits(x)


def make_weights(model: dict, seed: int) -> dict:
    """BF16 weights (uint16 bit patterns) in nn.Linear layout [out, in].

    Per layer: attn_norm [H] (None at encoder layer 0: that layer's attention
    norm is the identity), wqkv [3H, H], wo [H, H], mlp_norm [H],
    wup [2I, H] (first I rows feed GELU, last I rows are the gate),
    wdown [H, I]."""
    rng = np.random.default_rng(seed)
    H, I, V = model["hidden"], model["intermediate"], model["vocab"]
    w = {
        "tok_emb": _normal_bits(rng, (V, H), 0.02),
        "emb_norm": _normal_bits(rng, (H,), 0.02, 1.0),
        "final_norm": _normal_bits(rng, (H,), 0.02, 1.0),
        "layers": [],
    }
    L = model["n_encoder_layers"] + model["n_decision_layers"]
    for l in range(L):
        identity = l == 0 and model["first_attn_norm_identity"]
        w["layers"].append({
            "attn_norm": None if identity else _normal_bits(rng, (H,), 0.02, 1.0),
            "wqkv": _normal_bits(rng, (3 * H, H), 0.02),
            "wo": _normal_bits(rng, (H, H), 0.02),
            "mlp_norm": _normal_bits(rng, (H,), 0.02, 1.0),
            "wup": _normal_bits(rng, (2 * I, H), 0.02),
            "wdown": _normal_bits(rng, (H, I), 0.02),
        })
    return w


def make_inputs(model: dict, batch: int, seq: int, seed: int, length_range=None):
    """Token ids [batch, seq] int32 and row lengths [batch] int32."""
    rng = np.random.default_rng((seed, 1, batch, seq))
    ids = rng.integers(0, model["vocab"], size=(batch, seq), dtype=np.int64).astype(np.int32)
    if length_range is None:
        lengths = np.full((batch,), seq, np.int32)
    else:
        lo, hi = length_range
        lengths = rng.integers(lo, hi + 1, size=(batch,), dtype=np.int64).astype(np.int32)
    return ids, lengths


def workload(name: str):
    """(model, weights, ids, lengths) of a named workload."""
    model, B, S, seed, lr = WORKLOADS[name]
    return model, make_weights(model, seed), *make_inputs(model, B, S, seed, lr)


def weight_bytes(model: dict) -> int:
    """Bytes of the GEMM weights of all layers (the per-forward weight stream)."""
    H, I = model["hidden"], model["intermediate"]
    L = model["n_encoder_layers"] + model["n_decision_layers"]
    return 2 * L * (3 * H * H + H * H + 2 * I * H + H * I)
