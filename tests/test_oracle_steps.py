"""Pins of the oracle's single steps against closed forms, exact integer cases,
library routines and fp64 brute force (CPU only).

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, index or divisor, a transposed operand, swapped GeGLU halves, the
wrong window edge) makes it fail.
"""
import math

import numpy as np
import pytest
from scipy.special import erf

from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def ulp_bf16(v):
    """Spacing of BF16 numbers at |v| (2^(e-7) for v in [2^e, 2^(e+1)))."""
    v = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(v)) - 7)


# ------------------------------------------------------------------- BF16 --

@pytest.mark.parametrize("x,expect", [
    (1.0, 1.0),
    (1.0 + 2 ** -8, 1.0),                       # tie -> even (down)
    (1.0 + 3 * 2 ** -8, 1.0 + 2 ** -6),          # tie -> even (up)
    (1.0 + 2 ** -8 + 2 ** -20, 1.0 + 2 ** -7),   # above the tie
    (-(1.0 + 3 * 2 ** -8), -(1.0 + 2 ** -6)),
    (3.4e38, math.inf),                          # past the largest BF16 + half a step
    (0.0, 0.0),
    (2.0 ** -130, 2.0 ** -130),                  # subnormal, exact
])
def test_bf16_round_closed_form(orc, x, expect):
    assert orc.bf16_round(x) == expect


def test_bf16_round_nan_and_agreement(orc):
    assert math.isnan(orc.bf16_round(float("nan")))
    rng = np.random.default_rng(5)
    xs = (rng.standard_normal(2000) * 10.0 ** rng.integers(-20, 20, 2000)).astype(np.float32)
    ours = np.array([orc.bf16_round(float(v)) for v in xs], np.float32)
    # the seeded-input converter is an independent implementation of the same rounding
    np.testing.assert_array_equal(ours, bf16_bits_to_f32(f32_to_bf16_bits(xs)))


# -------------------------------------------------------------- LayerNorm --

def test_layernorm_constant_row_is_zero(orc):
    x = np.full((3, 256), 0.75, np.float32)
    y = bf16_bits_to_f32(orc.layernorm(bits(x), bits(np.ones(256)), 1e-5))
    assert np.all(y == 0.0)


def test_layernorm_alternating_closed_form(orc):
    # mean 0 and variance a^2 exactly; y = +-a / sqrt(a^2 + eps) * gamma
    a, n, eps = 0.5, 64, 1e-5
    x = np.array([a if i % 2 == 0 else -a for i in range(n)], np.float32)[None, :]
    gamma = np.linspace(0.5, 2.0, n).astype(np.float32)
    gb = bits(gamma)
    y = bf16_bits_to_f32(orc.layernorm(bits(x), gb, eps))[0]
    g = bf16_bits_to_f32(gb).astype(np.float64)
    expect = np.where(np.arange(n) % 2 == 0, 1.0, -1.0) * a / math.sqrt(a * a + eps) * g
    assert np.all(np.abs(y - expect) <= 0.5 * ulp_bf16(expect) + 1e-6 * np.abs(expect))
    # dividing by n - 1 instead of n would give |y| = sqrt((n-1)/n) * gamma: caught here
    assert np.abs(np.abs(y[0]) - g[0]) < 0.5 * ulp_bf16(g[0]) + 1e-6


def test_layernorm_power_of_two_scale_invariance(orc):
    rng = np.random.default_rng(0)
    x = bits(rng.standard_normal((4, 128)))
    xs = bits(bf16_bits_to_f32(x) * 4.0)
    g = bits(1 + 0.1 * rng.standard_normal(128))
    np.testing.assert_array_equal(orc.layernorm(x, g, 0.0), orc.layernorm(xs, g, 0.0))


def test_layernorm_fp64_brute_force(orc):
    rng = np.random.default_rng(1)
    x = bits(rng.standard_normal((16, 1024)) * 3 + 0.7)
    g = bits(1 + 0.02 * rng.standard_normal(1024))
    y = bf16_bits_to_f32(orc.layernorm(x, g, 1e-5)).astype(np.float64)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    gf = bf16_bits_to_f32(g).astype(np.float64)
    mu = xf.mean(1, keepdims=True)
    var = ((xf - mu) ** 2).mean(1, keepdims=True)
    ref = (xf - mu) / np.sqrt(var + 1e-5) * gf
    assert np.all(np.abs(y - ref) <= ulp_bf16(ref) * 0.5 + 1e-5 * np.abs(ref) + 1e-30)
    # the output has mean ~0 and variance ~1 before gamma (gamma ~ 1)
    assert np.abs(y.mean()) < 0.02 and abs(y.var() - 1.0) < 0.05


def test_embed_layernorm_gathers_rows(orc):
    rng = np.random.default_rng(2)
    emb = bits(rng.standard_normal((10, 64)))
    g = bits(np.ones(64))
    ids = np.array([3, 3, 9, 0], np.int32)
    x = orc.embed_layernorm(emb, g, ids, 1e-5)
    np.testing.assert_array_equal(x, orc.layernorm(emb[ids], g, 1e-5))
    np.testing.assert_array_equal(x[0], x[1])


# ----------------------------------------------------------------- Linear --

def test_linear_exact_on_integers(orc):
    rng = np.random.default_rng(3)
    x = rng.integers(-3, 4, (5, 7))
    w = rng.integers(-2, 3, (3, 7))     # [out, in]: a transpose would not even fit
    y = orc.linear_f32(bits(x), bits(w))
    np.testing.assert_array_equal(y, (x @ w.T).astype(np.float32))
    np.testing.assert_array_equal(orc.linear_f32(bits(x), bits(w), f64=True), y)


def test_linear_exact_long_k(orc):
    rng = np.random.default_rng(4)
    x = rng.integers(-8, 9, (3, 2624))
    w = rng.integers(-8, 9, (40, 2624))
    np.testing.assert_array_equal(orc.linear_f32(bits(x), bits(w)), (x @ w.T).astype(np.float32))


def test_linear_residual_and_plain_rounding(orc):
    rng = np.random.default_rng(5)
    x = rng.integers(-3, 4, (4, 16))
    w = rng.integers(-3, 4, (8, 16))
    r = rng.integers(-50, 50, (4, 8))
    y = bf16_bits_to_f32(orc.linear(bits(x), bits(w), orc.LINEAR_RESIDUAL, bits(r)))
    np.testing.assert_array_equal(y, (r + x @ w.T).astype(np.float32))
    # a non-representable sum is rounded once to BF16
    x1 = bits(np.array([[1.0, 2 ** -8]], np.float32))
    w1 = bits(np.array([[1.0, 1.0]], np.float32))
    assert bf16_bits_to_f32(orc.linear(x1, w1))[0, 0] == 1.0
    r1 = bits(np.array([[2 ** -8]], np.float32))
    # residual added before the single rounding: 1 + 2^-8 + 2^-8 = 1 + 2^-7 exactly
    assert bf16_bits_to_f32(orc.linear(x1, w1, orc.LINEAR_RESIDUAL, r1))[0, 0] == 1.0 + 2 ** -7


def gelu64(z):
    z = np.asarray(z, np.float64)
    return 0.5 * z * (1.0 + erf(z / math.sqrt(2.0)))


def test_gelu_special_values(orc):
    assert orc.gelu(0.0) == 0.0
    assert orc.gelu(10.0) == 10.0
    assert abs(orc.gelu(-10.0)) < 1e-20
    for z in np.linspace(-6, 6, 241):
        z = float(np.float32(z))
        # gelu(z) - gelu(-z) = z  (erf is odd)
        assert abs((orc.gelu(z) - orc.gelu(-z)) - z) <= 4e-7 * max(1.0, abs(z))
        assert abs(orc.gelu(z) - gelu64(z)) <= 4e-7 * max(1.0, abs(z))


def test_geglu_half_order(orc):
    # up-projection rows [0, I) feed GELU, rows [I, 2I) are the gate
    I, K = 6, 4
    rng = np.random.default_rng(6)
    h = bits(rng.standard_normal((3, K)))
    w_in = bits(rng.standard_normal((I, K)))
    w_gate = bits(rng.standard_normal((I, K)) * 0.5)
    y = bf16_bits_to_f32(orc.linear(h, np.concatenate([w_in, w_gate]), orc.LINEAR_GEGLU))
    hf, wi, wg = (bf16_bits_to_f32(a).astype(np.float64) for a in (h, w_in, w_gate))
    ref = gelu64(hf @ wi.T) * (hf @ wg.T)
    assert np.all(np.abs(y - ref) <= ulp_bf16(ref) * 0.5 + 1e-5 * np.abs(ref) + 1e-6)
    swapped = gelu64(hf @ wg.T) * (hf @ wi.T)
    assert np.max(np.abs(y - swapped)) > 0.05


# ------------------------------------------------------------------- RoPE --

@pytest.mark.parametrize("theta", [10000.0, 160000.0])
def test_rope_table_closed_forms(orc, theta):
    c, s = orc.rope_table(theta, 512, 32, bf16=True)
    assert np.all(c[0] == 1.0) and np.all(s[0] == 0.0)
    for p in (1, 2, 7, 100, 511):
        # pair 0 has frequency 1: angle = p
        assert c[p, 0] == orc.bf16_round(float(np.float32(math.cos(p))))
        assert s[p, 0] == orc.bf16_round(float(np.float32(math.sin(p))))
        # pair 16 of 32 has frequency theta^(-1/2)
        a = p / math.sqrt(theta)
        assert c[p, 16] == orc.bf16_round(float(np.float32(math.cos(a))))
        assert s[p, 16] == orc.bf16_round(float(np.float32(math.sin(a))))
    cf, sf = orc.rope_table(theta, 512, 32, bf16=False)
    assert np.max(np.abs(cf - c)) > 0 and np.all(np.abs(cf - c) <= 2.0 ** -9)
    assert cf[300, 31] == np.float32(math.cos(300 * theta ** (-62 / 64)))


def test_rope_identity_at_position_zero(orc):
    rng = np.random.default_rng(7)
    v = bf16_bits_to_f32(bits(rng.standard_normal(64)))
    c, s = orc.rope_table(10000.0, 4, 32)
    np.testing.assert_array_equal(orc.rope_vec(v, c[0], s[0]), v)


def test_rope_quarter_turn_pairs_and_signs(orc):
    rng = np.random.default_rng(8)
    v = bf16_bits_to_f32(bits(rng.standard_normal(64)))
    y = orc.rope_vec(v, np.zeros(32), np.ones(32))
    np.testing.assert_array_equal(y[:32], -v[32:])
    np.testing.assert_array_equal(y[32:], v[:32])


def test_rope_preserves_pair_norms(orc):
    rng = np.random.default_rng(9)
    c, s = orc.rope_table(160000.0, 512, 32, bf16=False)
    for p in (1, 63, 64, 511):
        v = bf16_bits_to_f32(bits(rng.standard_normal(64)))
        y = orc.rope_vec(v, c[p], s[p]).astype(np.float64)
        n0 = v[:32].astype(np.float64) ** 2 + v[32:].astype(np.float64) ** 2
        n1 = y[:32] ** 2 + y[32:] ** 2
        assert np.all(np.abs(np.sqrt(n1) - np.sqrt(n0)) <= 2.0 ** -7 * np.sqrt(n0) + 1e-6)


def test_rope_step_positions_and_v_untouched(orc):
    rng = np.random.default_rng(10)
    B, S, heads, D = 2, 5, 2, 64
    H = heads * D
    qkv = bits(rng.standard_normal((B * S, 3 * H)))
    c, s = orc.rope_table(10000.0, 512, 32)
    out = orc.rope(qkv, B, S, heads, D, c, s)
    np.testing.assert_array_equal(out[:, 2 * H:], qkv[:, 2 * H:])       # v untouched
    np.testing.assert_array_equal(out[0], qkv[0])                       # row 0, position 0
    np.testing.assert_array_equal(out[S], qkv[S])                       # row 1, position 0
    assert np.any(out[S + 1, :2 * H] != qkv[S + 1, :2 * H])
    qf = bf16_bits_to_f32(qkv)
    for t, p in ((3, 3), (S + 2, 2)):
        for base in (0, D, H, H + D):
            ref = orc.rope_vec(qf[t, base:base + D], c[p], s[p])
            np.testing.assert_array_equal(bf16_bits_to_f32(out[t, base:base + D]), ref)


# -------------------------------------------------------------- Attention --

def _pack(q, k, v):
    S, H = q.shape
    return bits(np.concatenate([q, k, v], axis=1))


def test_attention_single_key_returns_value(orc):
    rng = np.random.default_rng(11)
    S, H = 20, 64
    q, k, v = (rng.standard_normal((S, H)) for _ in range(3))
    qkv = _pack(q, k, v)
    ctx = orc.attention(qkv, [1], 1, S, 1, 64, True, 64)
    vb = bf16_bits_to_f32(qkv[:, 2 * H:])
    for i in range(S):
        np.testing.assert_array_equal(bf16_bits_to_f32(ctx[i]), vb[0])


@pytest.mark.parametrize("glob", [True, False])
def test_attention_uniform_scores_window_edges(orc, glob):
    # q = 0 makes every visible key equally likely: ctx[i][0] = mean of the
    # visible positions, ctx[i][1] = 1.  The mean pins both window edges.
    S, L, W, H = 200, 180, 64, 64
    q = np.zeros((S, H))
    k = np.random.default_rng(12).standard_normal((S, H))
    v = np.zeros((S, H))
    v[:, 0] = np.arange(S) / 4.0
    v[:, 1] = 1.0
    ctx = bf16_bits_to_f32(orc.attention(_pack(q, k, v), [L], 1, S, 1, 64, glob, W))
    for i in (0, 10, 63, 64, 65, 100, 150, 179, 190):
        lo, hi = (0, L) if glob else (max(0, i - W), min(L, i + W + 1))
        if lo >= hi:
            assert np.all(ctx[i] == 0.0)
            continue
        mean = (lo + hi - 1) / 2.0 / 4.0
        assert abs(ctx[i, 0] - mean) <= 0.5 * ulp_bf16(mean) + 1e-4, (i, ctx[i, 0], mean)
        assert ctx[i, 1] == 1.0


def test_attention_empty_key_rows_are_zero(orc):
    rng = np.random.default_rng(13)
    S, H = 150, 64
    qkv = _pack(*(rng.standard_normal((S, H)) for _ in range(3)))
    ctx = bf16_bits_to_f32(orc.attention(qkv, [10], 1, S, 1, 64, False, 64))
    assert np.all(ctx[74:] == 0.0) and np.all(ctx[:74] != 0.0)


def test_attention_fp64_brute_force(orc):
    rng = np.random.default_rng(14)
    B, S, heads, D, W = 2, 12, 2, 64, 3
    H = heads * D
    qkv = bits(rng.standard_normal((B * S, 3 * H)))
    lengths = [12, 7]
    for glob in (True, False):
        ctx = bf16_bits_to_f32(orc.attention(qkv, lengths, B, S, heads, D, glob, W))
        qf = bf16_bits_to_f32(qkv).astype(np.float64).reshape(B, S, 3, heads, D)
        for b in range(B):
            i = np.arange(S)[:, None]
            j = np.arange(S)[None, :]
            allowed = (j < lengths[b]) & (glob | (np.abs(i - j) <= W))
            for n in range(heads):
                sc = qf[b, :, 0, n] @ qf[b, :, 1, n].T / 8.0
                sc = np.where(allowed, sc, -np.inf)
                m = sc.max(1, keepdims=True)
                p = np.exp(sc - np.where(np.isfinite(m), m, 0))
                den = p.sum(1, keepdims=True)
                ref = np.where(den > 0, p / np.where(den > 0, den, 1), 0) @ qf[b, :, 2, n]
                got = ctx.reshape(B, S, heads, D)[b, :, n]
                assert np.all(np.abs(got - ref) <= 0.5 * ulp_bf16(ref) + 1e-5), (b, n, glob)
