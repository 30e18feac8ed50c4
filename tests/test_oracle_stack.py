"""Pins of the oracle's full stack (CPU only): structure tests with hand-made
weights whose output has a closed form, the layer schedule, and invariants
that any correct implementation of the definition satisfies bitwise
(padding, permutation, truncation, repeat)."""
import math

import numpy as np
import pytest

from transformer_encoder_bf16_gb300 import synth
from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, np.float32))


def tiny_model(**kw):
    m = dict(synth._COMMON, hidden=64, heads=1, head_dim=64, intermediate=64, vocab=16,
             n_encoder_layers=1, n_decision_layers=0, first_attn_norm_identity=0,
             final_norm=0)
    m.update(kw)
    return m


def zero_weights(m, rng, emb_scale=1.0):
    H, I, V = m["hidden"], m["intermediate"], m["vocab"]
    L = m["n_encoder_layers"] + m["n_decision_layers"]
    w = {"tok_emb": bits(rng.standard_normal((V, H)) * emb_scale),
         "emb_norm": bits(np.ones(H)), "final_norm": bits(np.ones(H)), "layers": []}
    for l in range(L):
        w["layers"].append({"attn_norm": bits(np.ones(H)), "wqkv": bits(np.zeros((3 * H, H))),
                            "wo": bits(np.zeros((H, H))), "mlp_norm": bits(np.ones(H)),
                            "wup": bits(np.zeros((2 * I, H))), "wdown": bits(np.zeros((H, I)))})
    return w


def ln64(x, g=1.0, eps=1e-5):
    x = np.asarray(x, np.float64)
    mu = x.mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(((x - mu) ** 2).mean(-1, keepdims=True) + eps) * g


def close(a, b, rel=2 ** -6):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.all(np.abs(a - b) <= rel * np.abs(b) + 1e-3)


def test_zero_weights_give_the_two_norms(orc):
    # all projections zero: out = LN_final(LN_emb(E[id])); decision layers add nothing
    m = tiny_model(n_encoder_layers=2, n_decision_layers=1, final_norm=1)
    rng = np.random.default_rng(0)
    w = zero_weights(m, rng, emb_scale=5.0)
    w["emb_norm"] = bits(np.full(64, 3.0))
    w["final_norm"] = bits(np.full(64, 0.5))
    ids = np.array([[1, 5, 7]], np.int32)
    out = orc.forward(m, w, ids, [3])[0]
    e = bf16_bits_to_f32(w["tok_emb"])[ids[0]]
    assert close(out, ln64(ln64(e, 3.0), 0.5))


def _identity_attention_layer(layer, H, c):
    # v = h, every other projection 0 except wo = c * I
    wqkv = np.zeros((3 * H, H))
    wqkv[2 * H:] = np.eye(H)
    layer["wqkv"] = bits(wqkv)
    layer["wo"] = bits(np.eye(H) * c)


def test_pre_norm_residual_attention(orc):
    # One token: attention returns v = h = LN(x), so x1 = x0 + c * LN(x0).
    # A post-norm layer would give LN(x0 + c x0) instead.
    m = tiny_model()
    rng = np.random.default_rng(1)
    w = zero_weights(m, rng)
    w["emb_norm"] = bits(np.full(64, 2.0))
    _identity_attention_layer(w["layers"][0], 64, 1.0)
    ids = np.array([[3]], np.int32)
    out = orc.forward(m, w, ids, [1])[0, 0]
    x0 = ln64(bf16_bits_to_f32(w["tok_emb"])[3], 2.0)
    assert close(out, x0 + ln64(x0))           # = 1.5 * x0
    assert not close(out, ln64(2 * x0))


def test_geglu_mlp_closed_form(orc):
    # attention contributes 0; a_in = alpha h, a_gate = beta h, down = I:
    # x1 = x0 + gelu(alpha h) * beta h, h = LN(x0)
    m = tiny_model()
    rng = np.random.default_rng(2)
    w = zero_weights(m, rng)
    alpha, beta = 1.5, 0.25
    w["layers"][0]["wup"] = bits(np.concatenate([np.eye(64) * alpha, np.eye(64) * beta]))
    w["layers"][0]["wdown"] = bits(np.eye(64))
    ids = np.array([[2, 9]], np.int32)
    out = orc.forward(m, w, ids, [2])[0]
    from scipy.special import erf
    x0 = ln64(bf16_bits_to_f32(w["tok_emb"])[ids[0]])
    h = ln64(x0)
    a = alpha * h
    assert close(out, x0 + 0.5 * a * (1 + erf(a / math.sqrt(2))) * beta * h)
    b = beta * h
    assert not close(out, x0 + 0.5 * b * (1 + erf(b / math.sqrt(2))) * alpha * h)


def test_final_norm_sits_between_encoder_and_decision_layers(orc):
    # encoder layer adds 0; x_f = LN(x0) * 3; decision layer adds LN(x_f) (v = h):
    # out = x_f + LN(x_f) = 4 * n.  A final norm after the decision layer would give 3 * n.
    m = tiny_model(n_encoder_layers=1, n_decision_layers=1, final_norm=1)
    rng = np.random.default_rng(3)
    w = zero_weights(m, rng)
    w["final_norm"] = bits(np.full(64, 3.0))
    _identity_attention_layer(w["layers"][1], 64, 1.0)
    out = orc.forward(m, w, np.array([[4]], np.int32), [1])[0, 0]
    n = ln64(ln64(bf16_bits_to_f32(w["tok_emb"])[4]))
    assert close(out, 4 * n)


def test_first_attention_norm_identity(orc):
    # with the identity reading, layer 0 projects x itself: x1 = x0 + c * x0 (no LN).
    m = tiny_model(first_attn_norm_identity=1)
    rng = np.random.default_rng(4)
    w = zero_weights(m, rng)
    w["emb_norm"] = bits(np.full(64, 2.0))
    w["layers"][0]["attn_norm"] = None
    _identity_attention_layer(w["layers"][0], 64, 1.0)
    out = orc.forward(m, w, np.array([[3]], np.int32), [1])[0, 0]
    x0 = ln64(bf16_bits_to_f32(w["tok_emb"])[3], 2.0)
    assert close(out, 2 * x0)


def _random_tiny(m, seed):
    return synth.make_weights(dict(m), seed)


def test_layer_schedule_global_every_third_and_decision_global(orc):
    # Output must depend on the local table exactly when some layer is local.
    base = tiny_model(n_encoder_layers=1, n_decision_layers=1, final_norm=1,
                      first_attn_norm_identity=1)
    ids, _ = synth.make_inputs(base, 1, 10, 0)
    for n_enc, expect_local in ((1, False), (3, True)):
        m = dict(base, n_encoder_layers=n_enc)
        w = _random_tiny(m, 5)
        a = orc.forward(m, w, ids, [10])
        b = orc.forward(dict(m, theta_local=777.0), w, ids, [10])
        c = orc.forward(dict(m, theta_global=777.0), w, ids, [10])
        assert np.array_equal(a, b) != expect_local, n_enc
        assert not np.array_equal(a, c)
    # global_every=1 makes every encoder layer global
    m = dict(base, n_encoder_layers=3, global_every=1)
    w = _random_tiny(m, 5)
    np.testing.assert_array_equal(orc.forward(m, w, ids, [10]),
                                  orc.forward(dict(m, theta_local=777.0), w, ids, [10]))


def test_local_window_limits_reach(orc):
    # A global layer carries a change of token 0 to every token; a local layer
    # with half window 2 carries it only to tokens 1 and 2.
    m = tiny_model(n_encoder_layers=1, local_half_window=2, first_attn_norm_identity=1)
    w = _random_tiny(m, 6)
    ids, _ = synth.make_inputs(m, 1, 10, 1)
    ids2 = ids.copy()
    ids2[0, 0] = (ids[0, 0] + 1) % m["vocab"]
    a = orc.forward(m, w, ids, [10])
    b = orc.forward(m, w, ids2, [10])
    assert not np.array_equal(a[0, 9], b[0, 9])      # global layer 0 reaches everything
    # two layers; layer 0's attention output is zeroed so that only the local
    # layer 1 mixes tokens
    m2 = tiny_model(n_encoder_layers=2, local_half_window=2, first_attn_norm_identity=1)
    w2 = _random_tiny(m2, 7)
    w2["layers"][0]["wo"] = bits(np.zeros((64, 64)))
    a = orc.forward(m2, w2, ids, [10])
    b = orc.forward(m2, w2, ids2, [10])
    assert np.array_equal(a[0, 3:], b[0, 3:])         # |i - 0| > 2: out of reach
    assert not np.array_equal(a[0, 2], b[0, 2])       # |i - 0| = 2: in reach


@pytest.fixture(scope="module")
def reduced():
    m = synth.REDUCED
    return m, synth.make_weights(m, 0)


def test_padding_does_not_change_valid_tokens(orc, reduced):
    m, w = reduced
    ids, _ = synth.make_inputs(m, 2, 150, 3)
    lengths = np.array([150, 70], np.int32)
    a = orc.forward(m, w, ids, lengths)
    ids2 = ids.copy()
    ids2[1, 70:] = (ids2[1, 70:] * 7 + 1) % m["vocab"]
    b = orc.forward(m, w, ids2, lengths)
    np.testing.assert_array_equal(a[1, :70], b[1, :70])
    np.testing.assert_array_equal(a[0], b[0])
    # truncating the padded row to its length gives the same valid tokens
    c = orc.forward(m, w, ids[1:, :70], lengths[1:])
    np.testing.assert_array_equal(a[1, :70], c[0])
    assert np.all(np.isfinite(a))


def test_row_permutation_and_repeat(orc, reduced):
    m, w = reduced
    ids, lengths = synth.make_inputs(m, 3, 40, 4, (5, 40))
    a = orc.forward(m, w, ids, lengths)
    perm = [2, 0, 1]
    b = orc.forward(m, w, ids[perm], lengths[perm])
    np.testing.assert_array_equal(a[perm], b)
    np.testing.assert_array_equal(a, orc.forward(m, w, ids, lengths))


def test_capture_and_rounding_floor(orc, reduced):
    # fp32 vs fp64 accumulation of the same definition: the spread sizes the
    # rounding floor two correct implementations can differ by.
    m, w = reduced
    ids, lengths = synth.make_inputs(m, 1, 48, 0)
    a, cap = orc.forward(m, w, ids, lengths, capture_layer=0)
    b = orc.forward(m, w, ids, lengths, accum_f64=True)
    assert np.all(np.isfinite(cap)) and not np.array_equal(cap, a)
    nrms = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert nrms < 5e-3
    assert np.all(bf16_bits_to_f32(f32_to_bf16_bits(a)) == a)     # BF16-valued output


def test_fp32_output_is_the_last_sum_before_rounding(orc, reduced):
    # Parity mode of the tolerance reading on hidden states: the last residual
    # sum comes back unrounded.  Rounding it to BF16 must give the default
    # output bit for bit, it must sit within half a BF16 step of it, and most
    # values must be off the BF16 grid (the rounding really is skipped).
    m, w = reduced
    ids, lengths = synth.make_inputs(m, 2, 40, 6, (9, 40))
    a = orc.forward(m, w, ids, lengths)
    f = orc.forward(m, w, ids, lengths, out_fp32=True)
    np.testing.assert_array_equal(bf16_bits_to_f32(f32_to_bf16_bits(f)), a)
    step = np.exp2(np.floor(np.log2(np.maximum(np.abs(a), 2.0 ** -120))) - 7)
    assert np.all(np.abs(f - a) <= 0.5 * step)
    assert np.mean(f != a) > 0.5
    # the layers before the last keep their BF16 storage points
    a2, c2 = orc.forward(m, w, ids, lengths, capture_layer=0)
    f2, d2 = orc.forward(m, w, ids, lengths, capture_layer=0, out_fp32=True)
    np.testing.assert_array_equal(c2, d2)


def test_fp32_output_with_zero_projections_is_the_norms(orc):
    # every projection zero: the last sum adds exactly 0 to a BF16 residual
    # stream, so the fp32 output equals the BF16 one
    m = tiny_model(n_encoder_layers=2, n_decision_layers=1, final_norm=1)
    w = zero_weights(m, np.random.default_rng(5), emb_scale=3.0)
    ids = np.array([[1, 4, 9, 2]], np.int32)
    np.testing.assert_array_equal(orc.forward(m, w, ids, [4], out_fp32=True),
                                  orc.forward(m, w, ids, [4]))


def test_rejects_bad_arguments(orc, reduced):
    m, w = reduced
    ids, _ = synth.make_inputs(m, 1, 8, 0)
    with pytest.raises(ValueError):
        orc.forward(m, w, ids, [9])                # length > S
    with pytest.raises(ValueError):
        orc.forward(m, w, ids, [0])                # empty row
    bad = ids.copy()
    bad[0, 0] = m["vocab"]
    with pytest.raises(ValueError):
        orc.forward(m, w, bad, [8])                # id out of range


def _embedding(orc, m, w, ids):
    B, S = ids.shape
    x = orc.embed_layernorm(w["tok_emb"], w["emb_norm"], ids, m["ln_eps"])
    return bf16_bits_to_f32(x).reshape(B, S, m["hidden"])


@pytest.mark.parametrize("accum_f64,out_fp32", [(False, False), (True, False), (False, True)])
def test_layer_chain_reproduces_forward(orc, reduced, accum_f64, out_fp32):
    # One layer at a time from the embedding output (the final norm taken
    # inside the first decision layer) must give the whole stack bit for bit;
    # a layer that ignored its input, or applied the final norm at the wrong
    # layer, breaks the chain.
    m, w = reduced
    ids, lengths = synth.make_inputs(m, 2, 40, 8, (7, 40))
    ref = orc.forward(m, w, ids, lengths, accum_f64=accum_f64, out_fp32=out_fp32)
    x = _embedding(orc, m, w, ids)
    L = m["n_encoder_layers"] + m["n_decision_layers"]
    for l in range(L):
        nxt = orc.layer(m, w, l, x, lengths, accum_f64=accum_f64, out_fp32=out_fp32)
        assert not np.array_equal(nxt, x)
        x = nxt
    np.testing.assert_array_equal(x, ref)


def test_layer_matches_the_captured_stream(orc, reduced):
    m, w = reduced
    ids, lengths = synth.make_inputs(m, 1, 24, 9)
    _, c1 = orc.forward(m, w, ids, lengths, capture_layer=1)
    _, c2 = orc.forward(m, w, ids, lengths, capture_layer=2)
    np.testing.assert_array_equal(orc.layer(m, w, 2, c1, lengths), c2)


def test_layer_rejects_bad_arguments(orc, reduced):
    m, w = reduced
    x = np.zeros((1, 8, m["hidden"]), np.float32)
    with pytest.raises(ValueError):
        orc.layer(m, w, m["n_encoder_layers"] + m["n_decision_layers"], x, [8])  # no such layer
    with pytest.raises(ValueError):
        orc.layer(m, w, 0, x, [9])                                               # length > S
    with pytest.raises(ValueError):                                              # final norm missing
        orc.layer(m, dict(w, final_norm=None), m["n_encoder_layers"], x, [8])
