"""The marker-row last layer ("perf(model): exact Metal speed-ups of the
forward pass - #45": keys and values need every position, but everything
after them is row-wise and attention is independent per query row, so the
last layer attends from, projects and runs its MLP on the marker rows alone),
and its subset-query attention entry point.

The oracle side is the plain definition: the full last layer, then the
marker rows selected.  The subset attention is checked against the matching
rows of full attention (1, 2 and 3 rows, as the page's own test does), the
marker forward against the full forward's rows and against the oracle's last
layer fed the GPU's own state entering it (teacher-forced, the pages' nRMS
5e-3), and the argument errors (a marker on padding is a client error)."""
import numpy as np
import pytest

import oracle
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth
from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32

from gpu_util import i32_dev, nrms, require_gpu, rnd_bits, to_bits, to_dev, ulp_bf16

pytestmark = pytest.mark.gpu

NRMS_LIMIT = 5e-3


@pytest.mark.parametrize("B,S,heads,lengths,glob,hw,pos", [
    (1, 48, 16, [48], True, 64, [[5]]),
    (1, 48, 16, [48], True, 64, [[0, 47]]),
    (2, 200, 4, [200, 77], True, 64, [[3, 150, 199], [76, 0, 40]]),
    (2, 200, 4, [200, 77], False, 64, [[3, 150, 199], [76, 0, 40]]),
    (3, 130, 2, [130, 1, 65], False, 3, [[129, 64], [0, 0], [64, 1]]),
    (4, 512, 16, [512, 300, 33, 450], True, 64, [list(range(0, 33, 1))] * 4),
])
def test_subset_attention_equals_rows_of_full_attention(B, S, heads, lengths, glob, hw, pos):
    torch = require_gpu()
    rng = np.random.default_rng(B * S + heads)
    H = heads * 64
    lengths = np.array(lengths, np.int32)
    pos = np.array(pos, np.int32)
    kmax = pos.shape[1]
    qkv = rnd_bits(rng, (B * S, 3 * H), std=0.7)
    q_tok = (np.arange(B)[:, None] * S + pos).astype(np.int32).reshape(-1)
    dq = to_dev(qkv)
    full = torch.empty((B * S, H), dtype=torch.bfloat16, device="cuda")
    te.attention(dq, i32_dev(lengths), B, S, heads, glob, hw, full)
    rows = torch.full((B * kmax, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    te.attention_rows(dq, i32_dev(lengths), i32_dev(q_tok), i32_dev(pos.reshape(-1)), B, S, kmax,
                      heads, glob, hw, rows)
    torch.cuda.synchronize()
    got = to_bits(rows)
    # same arithmetic as the full kernel: the matching rows bit for bit
    np.testing.assert_array_equal(got, to_bits(full)[q_tok])
    # and the oracle's rows within the attention tolerance of the step tests
    ref = bf16_bits_to_f32(oracle.attention(qkv, lengths, B, S, heads, 64, glob, hw))[q_tok]
    g = bf16_bits_to_f32(got).astype(np.float64)
    v = bf16_bits_to_f32(qkv).reshape(B, S, 3, heads, 64)[:, :, 2]
    for m, t in enumerate(q_tok):
        b = t // S
        vmax = np.abs(v[b, :lengths[b]]).max(axis=(0, 2))
        lim = 0.5 * ulp_bf16(ref[m]) + 2.0 ** -8 * np.repeat(vmax, 64)
        assert np.all(np.abs(g[m] - ref[m]) <= lim), (m, float(np.max(np.abs(g[m] - ref[m]) - lim)))


def _markers(lengths, kmax, rng, empty=0):
    pos = np.full((len(lengths), kmax), -1, np.int32)
    for b, L in enumerate(lengths):
        k = max(1, kmax - empty)
        pos[b, :k] = rng.choice(int(L), size=min(k, int(L)), replace=False).tolist() + \
            [0] * (k - min(k, int(L)))
    return pos


_enc = {}


def encoder(name):
    model, B, S, seed, lr = synth.WORKLOADS[name]
    if name not in _enc:
        _enc.clear()
        w = synth.make_weights(model, seed)
        _enc[name] = (w, te.Encoder(model, te.upload_weights(w)))
    return (model, B, S, seed, lr) + _enc[name]


@pytest.mark.parametrize("name,kmax,empty", [
    ("reduced_1x48", 1, 0), ("reduced_1x48", 3, 0), ("full_1x48", 2, 0), ("full_4x64", 3, 1),
    ("full_4x464", 4, 0), ("full_16x512", 128, 0), ("full_16x512", 8, 3),
])
def test_marker_forward_matches_full_forward_and_oracle_last_layer(name, kmax, empty):
    torch = require_gpu()
    model, B, S, seed, lr, w, enc = encoder(name)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    pos = _markers(lengths, kmax, np.random.default_rng(kmax), empty)
    H = model["hidden"]
    L = model["n_encoder_layers"] + model["n_decision_layers"]
    out = torch.empty((B, S, H), dtype=torch.bfloat16, device="cuda")
    states = torch.empty((L, B, S, H), dtype=torch.bfloat16, device="cuda")
    enc.debug_capture(ids, lengths, out, states)
    mk = torch.full((B * kmax, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    enc.run_markers(ids, lengths, pos, mk)
    enc.check()
    got = bf16_bits_to_f32(to_bits(mk)).reshape(B, kmax, H).astype(np.float64)
    full = bf16_bits_to_f32(to_bits(out)).reshape(B, S, H)
    x_last = bf16_bits_to_f32(to_bits(states))[L - 1]
    assert np.all(np.isfinite(got))                       # empty slots too
    gs, fs, rs = [], [], []
    for b in range(B):
        n = int(lengths[b])
        ref = oracle.layer(model, w, L - 1, x_last[b:b + 1, :n], lengths[b:b + 1])[0]
        for j in range(kmax):
            p = pos[b, j]
            if p < 0:
                continue
            gs.append(got[b, j])
            fs.append(full[b, p])
            rs.append(ref[p])
    g, f, r = (np.array(a, np.float64) for a in (gs, fs, rs))
    e_full, e_orc = nrms(g, f), nrms(g, r)
    print(f"\n[markers] {name} kmax={kmax}: vs full forward rows nRMS {e_full:.2e}, vs oracle last "
          f"layer (teacher-forced) nRMS {e_orc:.2e}, max|d| {np.max(np.abs(g - r)):.2e}")
    assert e_full <= NRMS_LIMIT and e_orc <= NRMS_LIMIT, (e_full, e_orc)
    # repeat through the captured graph of this (batch, seq, kmax): same bytes
    mk2 = torch.empty_like(mk)
    enc.run_markers(ids, lengths, pos, mk2)
    enc.check()
    np.testing.assert_array_equal(to_bits(mk2), to_bits(mk))


def test_marker_arguments_are_checked():
    torch = require_gpu()
    model, B, S, seed, lr, w, enc = encoder("full_4x64")
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    H = model["hidden"]
    out = torch.empty((B * 4, H), dtype=torch.bfloat16, device="cuda")
    bad = np.zeros((B, 4), np.int32)
    bad[1, 2] = lengths[1]                        # a marker on padding
    with pytest.raises(te.LayaError) as ex:
        enc.run_markers(ids, lengths, bad, out)
    assert ex.value.code == te.E_INVAL
    bad[1, 2] = -2
    with pytest.raises(te.LayaError):
        enc.run_markers(ids, lengths, bad, out)
    big = np.zeros((B, 513), np.int32)            # B * kmax > 2048
    with pytest.raises(te.LayaError):
        enc.run_markers(ids, lengths, big, torch.empty((B * 513, H), dtype=torch.bfloat16,
                                                       device="cuda"))
    # the handle is not poisoned by argument errors
    enc.run_markers(ids, lengths, np.zeros((B, 4), np.int32), out)
    enc.check()
