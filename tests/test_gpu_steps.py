"""Per-step parity of the CUDA kernels against the CPU oracle, through the C
ABI (laya_op_*), on seeded inputs at sizes that span several tiles and ragged
tails.  RoPE must be bit-exact; LayerNorm and the projections may differ from
the oracle's sequential fp32 sums by one BF16 step where the fp32 value sits
next to a rounding boundary; attention is bounded by the BF16 rounding of the
probabilities fed to the P.V product."""
import numpy as np
import pytest

import oracle
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits

from gpu_util import bf16_close, i32_dev, nrms, require_gpu, rnd_bits, to_bits, to_dev, ulp_bf16

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------------ GEMM --

@pytest.mark.parametrize("M,N,K,splits,nt", [
    (48, 256, 128, 1, 0), (48, 384, 1024, 4, 0), (7, 128, 256, 2, 16), (300, 520, 192, 3, 0),
    (513, 136, 64, 1, 256), (100, 1024, 2624, 8, 0),
    # persistent kernel: several tiles per CTA, both TMEM accumulators, ragged edges
    (2000, 1024, 128, 1, 32), (3000, 520, 256, 1, 48), (1111, 3072, 1024, 1, 0)])
def test_linear_exact_integers(M, N, K, splits, nt):
    # small integers: every partial sum is exact in fp32, so any layout,
    # swizzle, transpose or split-K error shows up as a wrong value
    torch = require_gpu()
    rng = np.random.default_rng(M * 7 + N)
    x = rng.integers(-3, 4, (M, K)).astype(np.float32)
    w = rng.integers(-2, 3, (N, K)).astype(np.float32)
    xb, wb = f32_to_bf16_bits(x), f32_to_bf16_bits(w)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    te.linear(to_dev(xb), to_dev(wb), y, te.KIND_PLAIN, splits=splits, tile_tokens=nt)
    torch.cuda.synchronize()
    ref = (x.astype(np.int64) @ w.astype(np.int64).T).astype(np.float32)
    np.testing.assert_array_equal(bf16_bits_to_f32(to_bits(y)), bf16_bits_to_f32(f32_to_bf16_bits(ref)))


@pytest.mark.parametrize("kind", [te.KIND_PLAIN, te.KIND_RESIDUAL, te.KIND_GEGLU])
@pytest.mark.parametrize("M,N,K,splits,nt", [
    (48, 3072, 1024, 0, 0), (48, 1024, 2624, 0, 0), (1, 2624, 1024, 0, 0), (256, 1024, 1024, 0, 0),
    (464, 1024, 1024, 3, 0), (600, 640, 256, 1, 128), (130, 2624, 1024, 2, 48),
    (1200, 3072, 1024, 1, 0), (1000, 1024, 2624, 1, 112), (48, 1024, 2624, 16, 48),
    (48, 1024, 1024, 12, 48), (100, 640, 1024, 16, 64)])
def test_linear_matches_oracle(kind, M, N, K, splits, nt):
    torch = require_gpu()
    rng = np.random.default_rng(1000 + M + N + K + kind)
    Nw = 2 * N if kind == te.KIND_GEGLU else N
    xb = rnd_bits(rng, (M, K))
    wb = rnd_bits(rng, (Nw, K), std=0.02)
    rb = rnd_bits(rng, (M, N), std=2.0) if kind == te.KIND_RESIDUAL else None
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    r_dev = to_dev(rb) if rb is not None else None
    te.linear(to_dev(xb), to_dev(wb), y, kind, residual=r_dev, splits=splits, tile_tokens=nt)
    torch.cuda.synchronize()
    ref = oracle.linear(xb, wb, kind, rb)
    ok, msg = bf16_close(to_bits(y), ref, ulps=1.0, min_exact=0.97)
    assert ok, msg


@pytest.mark.parametrize("kind", [te.KIND_PLAIN, te.KIND_RESIDUAL, te.KIND_GEGLU])
@pytest.mark.parametrize("M,N,K,nt", [
    (2000, 1024, 1024, 224), (4117, 2624, 1024, 128), (1111, 520, 256, 64), (300, 3072, 1024, 48),
    (8192, 1024, 2624, 224)])
def test_linear_paired_equals_unpaired_and_oracle(kind, M, N, K, nt):
    # the persistent kernel in clusters of two (the token tile, or the weight
    # tiles, multicast into both CTAs) computes every tile exactly as the
    # single-CTA kernel: bit for bit, twice in a row; odd feature- and
    # token-tile counts (2624 / 128, 520 / 128, 4117 / 128 ...) leave the last
    # pair's second tile past N or past the tokens
    torch = require_gpu()
    rng = np.random.default_rng(2000 + M + N + K + kind)
    if kind == te.KIND_GEGLU:
        nt = min(nt, 128)   # two accumulators, double-buffered: 4 x nt <= 512 TMEM columns
    Nw = 2 * N if kind == te.KIND_GEGLU else N
    xb = rnd_bits(rng, (M, K))
    wb = rnd_bits(rng, (Nw, K), std=0.02)
    rb = rnd_bits(rng, (M, N), std=2.0) if kind == te.KIND_RESIDUAL else None
    r_dev = to_dev(rb) if rb is not None else None
    outs = []
    for paired in (0, 1, 1, 2, 2, 3, 3):
        y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        te.linear(to_dev(xb), to_dev(wb), y, kind, residual=r_dev, splits=1, tile_tokens=nt,
                  paired=paired)
        torch.cuda.synchronize()
        outs.append(to_bits(y))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])
    if M <= 2000:
        ok, msg = bf16_close(outs[1], oracle.linear(xb, wb, kind, rb), ulps=1.0, min_exact=0.97)
        assert ok, msg


@pytest.mark.parametrize("M,N,K,nt", [
    (4117, 2624, 1024, 240), (4117, 2624, 1024, 128), (1111, 576, 256, 64), (300, 3072, 1024, 48),
    (48, 2624, 1024, 48), (8192, 1024, 2624, 256), (1, 64, 64, 16)])
def test_linear_geglu_interleaved_equals_geglu(M, N, K, nt):
    # one 128-row weight tile holding 64 rows of each half (read through a 4-D
    # tensor map) gives the two-tile GeGLU's values bit for bit: the same fp32
    # accumulators meet in the same epilogue arithmetic; also in both pairings
    torch = require_gpu()
    rng = np.random.default_rng(3000 + M + N + K)
    xb = rnd_bits(rng, (M, K))
    wb = rnd_bits(rng, (2 * N, K), std=0.02)
    x_dev, w_dev = to_dev(xb), to_dev(wb)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    te.linear(x_dev, w_dev, y, te.KIND_GEGLU, splits=1, tile_tokens=min(nt, 128))
    torch.cuda.synchronize()
    ref = to_bits(y)
    for paired in (0, 0, 1, 2, 3):
        y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
        te.linear(x_dev, w_dev, y, te.KIND_GEGLU_IL, splits=1, tile_tokens=nt, paired=paired)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_bits(y), ref)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    te.linear_noalloc(x_dev, w_dev, y, te.KIND_GEGLU_IL, splits=1, tile_tokens=nt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(y), ref)
    if M <= 1111:
        ok, msg = bf16_close(ref, oracle.linear(xb, wb, te.KIND_GEGLU, None), ulps=1.0,
                             min_exact=0.97)
        assert ok, msg


def test_linear_geglu_interleaved_rejects_what_it_cannot_run():
    torch = require_gpu()
    x = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2 * 96, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((64, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(te.LayaError):   # N not a multiple of 64
        te.linear(x, w, y, te.KIND_GEGLU_IL, splits=1)
    w = torch.zeros((2 * 128, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(te.LayaError):   # split-K is not offered
        te.linear(x, w, y, te.KIND_GEGLU_IL, splits=2)
    with pytest.raises(te.LayaError):   # nor LayerNorm on load (split kernel only)
        te.linear_ln(x, torch.ones(256, dtype=torch.bfloat16, device="cuda"), 1e-5, w, y,
                     te.KIND_GEGLU_IL)


def test_linear_residual_in_place_and_repeat():
    torch = require_gpu()
    rng = np.random.default_rng(7)
    M, N, K = 48, 1024, 1024
    xb, wb, rb = rnd_bits(rng, (M, K)), rnd_bits(rng, (N, K), 0.02), rnd_bits(rng, (M, N))
    ref = oracle.linear(xb, wb, te.KIND_RESIDUAL, rb)
    outs = []
    for _ in range(2):
        y = to_dev(rb)
        te.linear(to_dev(xb), to_dev(wb), y, te.KIND_RESIDUAL, residual=y)
        torch.cuda.synchronize()
        outs.append(to_bits(y))
    np.testing.assert_array_equal(outs[0], outs[1])          # deterministic split-K
    ok, msg = bf16_close(outs[0], ref, ulps=1.0, min_exact=0.97)
    assert ok, msg


def test_linear_plan_small_shapes_fill_the_gpu():
    require_gpu()
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for (N, K, kind) in ((3072, 1024, 0), (1024, 1024, 1), (2624, 1024, 2), (1024, 2624, 1)):
        nt, splits, ctas = te.linear_plan(48, K, N, kind, sms)
        assert nt <= 48 and ctas >= sms // 3, (N, K, nt, splits, ctas)


# ------------------------------------------------------------- row steps --

@pytest.mark.parametrize("M,H", [(1, 256), (7, 1024), (300, 1024), (48, 256), (1000, 2048)])
def test_layernorm_matches_oracle(M, H):
    torch = require_gpu()
    rng = np.random.default_rng(M + H)
    xb = rnd_bits(rng, (M, H), std=2.0, mean=0.3)
    gb = rnd_bits(rng, (H,), std=0.02, mean=1.0)
    y = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    te.layernorm(to_dev(xb), to_dev(gb), 1e-5, y)
    x_in = to_dev(xb)
    te.layernorm(x_in, to_dev(gb), 1e-5, x_in)                 # in place
    torch.cuda.synchronize()
    ref = oracle.layernorm(xb, gb, 1e-5)
    ok, msg = bf16_close(to_bits(y), ref, ulps=1.0, min_exact=0.98)
    assert ok, msg
    np.testing.assert_array_equal(to_bits(x_in), to_bits(y))


def test_embed_layernorm_matches_oracle_and_flags_bad_ids():
    torch = require_gpu()
    rng = np.random.default_rng(3)
    V, H, M = 4096, 1024, 333
    eb = rnd_bits(rng, (V, H), std=0.02)
    gb = rnd_bits(rng, (H,), std=0.02, mean=1.0)
    ids = rng.integers(0, V, M).astype(np.int32)
    x = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    te.embed_layernorm(to_dev(eb), to_dev(gb), i32_dev(ids), 1e-5, x, err_dev=err)
    torch.cuda.synchronize()
    ok, msg = bf16_close(to_bits(x), oracle.embed_layernorm(eb, gb, ids, 1e-5), 1.0, 0.98)
    assert ok, msg
    assert int(err[0]) == 0
    bad = ids.copy()
    bad[5] = V
    te.embed_layernorm(to_dev(eb), to_dev(gb), i32_dev(bad), 1e-5, x, err_dev=err)
    torch.cuda.synchronize()
    assert int(err[0]) != 0


@pytest.mark.parametrize("theta", [10000.0, 160000.0])
@pytest.mark.parametrize("B,S,heads", [(1, 48, 16), (4, 64, 16), (2, 129, 4), (16, 512, 16)])
def test_rope_bit_exact(theta, B, S, heads):
    torch = require_gpu()
    rng = np.random.default_rng(B * S + heads)
    H = heads * 64
    qkv = rnd_bits(rng, (B * S, 3 * H), std=0.7)
    c, s = te.rope_table(theta, 512, 32)
    dev = to_dev(qkv)
    te.rope(dev, torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), B, S, heads)
    torch.cuda.synchronize()
    got = to_bits(dev)
    ref = oracle.rope(qkv, B, S, heads, 64, *oracle.rope_table(theta, 512, 32))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(got[:, 2 * H:], qkv[:, 2 * H:])   # V bytes preserved


def _attention_case(B, S, heads, lengths, glob, hw, seed, impl="mma"):
    torch = require_gpu()
    rng = np.random.default_rng(seed)
    H = heads * 64
    qkv = rnd_bits(rng, (B * S, 3 * H), std=0.7)
    ctx = torch.full((B * S, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn = te.attention if impl == "mma" else te.attention_tc
    fn(to_dev(qkv), i32_dev(lengths), B, S, heads, glob, hw, ctx)
    torch.cuda.synchronize()
    got = bf16_bits_to_f32(to_bits(ctx)).reshape(B, S, H)
    ref = bf16_bits_to_f32(oracle.attention(qkv, lengths, B, S, heads, 64, glob, hw)).reshape(B, S, H)
    v = bf16_bits_to_f32(qkv).reshape(B, S, 3, heads, 64)[:, :, 2]
    for b in range(B):
        L = lengths[b]
        g, r = got[b, :L].astype(np.float64), ref[b, :L].astype(np.float64)
        vmax = np.abs(v[b, :L]).max(axis=(0, 2))                     # per head
        lim = 0.5 * ulp_bf16(r) + 2.0 ** -8 * np.repeat(vmax, 64)[None, :]
        assert np.all(np.abs(g - r) <= lim), (b, float(np.max(np.abs(g - r) - lim)))
        assert nrms(g, r) < 3e-3
    assert np.all(np.isfinite(got))                                   # padded rows too


@pytest.mark.parametrize("B,S,heads,lengths,glob,hw", [
    (1, 48, 16, [48], True, 64),
    (4, 64, 16, [16, 64, 33, 50], False, 64),
    (2, 200, 4, [200, 77], False, 64),
    (2, 200, 4, [200, 77], True, 64),
    (1, 512, 16, [512], False, 64),
    (3, 130, 2, [130, 1, 65], False, 64),
    (3, 130, 2, [130, 1, 65], True, 64),
    (2, 300, 2, [300, 129], False, 3),
    (2, 464, 4, [464, 300], False, 128),
])
@pytest.mark.parametrize("impl", ["mma", "tc"])
def test_attention_matches_oracle(B, S, heads, lengths, glob, hw, impl):
    _attention_case(B, S, heads, np.array(lengths, np.int32), glob, hw, seed=B * S + heads, impl=impl)


@pytest.mark.parametrize("B,S,heads,lengths,glob,theta", [
    (1, 48, 16, [48], True, 160000.0),
    (4, 64, 16, [16, 64, 33, 50], False, 10000.0),
    (2, 200, 4, [200, 77], False, 10000.0),
    (3, 130, 2, [130, 1, 65], True, 160000.0),
    (2, 512, 2, [512, 300], True, 160000.0),
])
def test_attention_with_fused_rope_matches_oracle(B, S, heads, lengths, glob, theta):
    # the fused kernel rotates q and k in shared memory; the oracle applies
    # RoPE to the packed projection first and then attends
    torch = require_gpu()
    rng = np.random.default_rng(B * S + heads + 7)
    H = heads * 64
    lengths = np.array(lengths, np.int32)
    qkv = rnd_bits(rng, (B * S, 3 * H), std=0.7)
    c, s = te.rope_table(theta, 512, 32)
    dev = to_dev(qkv)
    ctx = torch.full((B * S, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    te.attention_rope(dev, i32_dev(lengths), torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(),
                      B, S, heads, glob, 64, ctx)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(dev), qkv)                  # projection not modified
    rotated = oracle.rope(qkv, B, S, heads, 64, *oracle.rope_table(theta, 512, 32))
    ref = bf16_bits_to_f32(oracle.attention(rotated, lengths, B, S, heads, 64, glob, 64)).reshape(B, S, H)
    got = bf16_bits_to_f32(to_bits(ctx)).reshape(B, S, H)
    v = bf16_bits_to_f32(qkv).reshape(B, S, 3, heads, 64)[:, :, 2]
    for b in range(B):
        L = lengths[b]
        g, r = got[b, :L].astype(np.float64), ref[b, :L].astype(np.float64)
        vmax = np.abs(v[b, :L]).max(axis=(0, 2))
        lim = 0.5 * ulp_bf16(r) + 2.0 ** -8 * np.repeat(vmax, 64)[None, :]
        assert np.all(np.abs(g - r) <= lim), (b, float(np.max(np.abs(g - r) - lim)))
        assert nrms(g, r) < 3e-3
    assert np.all(np.isfinite(got))


@pytest.mark.parametrize("B,S,splits,nt,theta", [
    (1, 48, 0, 0, 160000.0),        # library plan (split-K clusters at 48 tokens)
    (4, 64, 4, 64, 10000.0),        # forced split-K
    (1, 48, 16, 48, 10000.0),       # split-K cluster of 16 (RoPE tiles: some ranks reduce nothing)
    (1, 48, 12, 48, 160000.0),      # uneven slices
    (2, 300, 1, 112, 10000.0),      # persistent kernel, several tiles per CTA
    (16, 512, 0, 0, 160000.0),      # library plan at 8192 tokens
])
def test_qkv_with_rope_epilogue_bit_exact(B, S, splits, nt, theta):
    # RoPE applied in the QKV epilogue must equal the plain projection followed
    # by the stand-alone RoPE kernel, byte for byte (q and k rotated, v as is)
    torch = require_gpu()
    rng = np.random.default_rng(B * S + splits)
    H, M = 1024, B * S
    xb, wb = rnd_bits(rng, (M, H)), rnd_bits(rng, (3 * H, H), std=0.02)
    c, s = te.rope_table(theta, 512, 32)
    cd, sd = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
    x, w = to_dev(xb), to_dev(wb)
    fused = torch.empty((M, 3 * H), dtype=torch.bfloat16, device="cuda")
    te.linear_rope(x, w, fused, cd, sd, S, 2 * H, splits=splits, tile_tokens=nt)
    plain = torch.empty_like(fused)
    te.linear(x, w, plain, te.KIND_PLAIN, splits=splits, tile_tokens=nt)
    two_step = plain.clone()
    te.rope(two_step, cd, sd, B, S, 16)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(fused), to_bits(two_step))
    np.testing.assert_array_equal(to_bits(fused)[:, 2 * H:], to_bits(plain)[:, 2 * H:])


@pytest.mark.parametrize("kind", [te.KIND_PLAIN, te.KIND_GEGLU])
@pytest.mark.parametrize("M,N,splits,nt", [(48, 3072, 4, 48), (48, 2624, 6, 48), (256, 1024, 2, 128),
                                           (100, 640, 3, 112), (48, 1024, 1, 48), (48, 1024, 16, 48)])
def test_linear_with_layernorm_on_load_bit_exact(kind, M, N, splits, nt):
    # the GEMM normalising its input tiles on load equals the LayerNorm kernel
    # followed by the same GEMM plan, byte for byte
    torch = require_gpu()
    rng = np.random.default_rng(M + N + splits + kind)
    K = 1024
    Nw = 2 * N if kind == te.KIND_GEGLU else N
    xb = rnd_bits(rng, (M, K), std=1.5, mean=0.2)
    gb = rnd_bits(rng, (K,), std=0.02, mean=1.0)
    wb = rnd_bits(rng, (Nw, K), std=0.02)
    x, g, w = to_dev(xb), to_dev(gb), to_dev(wb)
    fused = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    te.linear_ln(x, g, 1e-5, w, fused, kind, splits=splits, tile_tokens=nt)
    h = torch.empty_like(x)
    te.layernorm(x, g, 1e-5, h)
    two_step = torch.empty_like(fused)
    te.linear(h, w, two_step, kind, splits=splits, tile_tokens=nt)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_bits(fused), to_bits(two_step))
    ref = oracle.linear(oracle.layernorm(xb, gb, 1e-5), wb, kind)
    ok, msg = bf16_close(to_bits(fused), ref, ulps=1.0, min_exact=0.9)
    assert ok, msg
