"""Full-stack parity of laya_enc_run against the CPU oracle, and the stack
invariants the GPU path must keep bitwise (repeat, eager vs graph, padding,
row order, reused workspaces), through the C ABI.

Tolerances.  "[Performance]: Optimize native Rust/CUDA Laya inference #66"
("Starting evidence") keeps an nRMS limit of 5e-3 on hidden states.  With the
synthetic N(0, 0.02) weights, the definition itself spreads further than that
at full depth: the oracle run with fp32 sums and with fp64 sums (two correct
evaluations of the same definition, differing only in rounding) drift apart
by about 6e-4 nRMS per layer (7e-4 after layer 0, 3.6e-3 after layer 3,
1.8e-2 after layer 29 at 1 x 48), because every BF16 storage point turns an
fp32 ordering difference into a one-step flip that the residual stream keeps.
So:
  * depth prefix (layers 0-3: global, local, local, global): nRMS <= 5e-3,
    the pages' limit as written;
  * full depth: the GPU must be no farther from the fp64-summed oracle than
    the fp32-summed oracle is (nRMS within 1.5x; max-abs within 2x plus one
    BF16 step of the largest reference magnitude), and within 2x of that
    floor from the fp32 oracle;
  * every layer alone, fed the GPU's own input state (tests/test_gpu_layers.py):
    nRMS <= 5e-3 as written, on every row of every workload.
The 2e-3 max-abs figure of "[RFC]: Native Laya inference with Rust and CUDA
#14" bounded decision outputs; on BF16 hidden states of magnitude 2..8 a
single BF16 step is 1.6e-2..3.1e-2, so it is reported, not asserted."""
import os
import time

import numpy as np
import pytest

import oracle
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth
from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32

from gpu_util import i32_dev, nrms, require_gpu, to_bits, ulp_bf16

pytestmark = pytest.mark.gpu

NRMS_LIMIT = 5e-3

_cache = {}


def encoder_for(model, seed, n_layers=None):
    """(host weights, Encoder).  n_layers truncates the stack to its first
    n_layers encoder layers (no decision layers, no final norm): the output
    is then the residual stream after layer n_layers - 1."""
    key = (model["name"], seed)
    if key not in _cache:
        _cache.clear()
        w = synth.make_weights(model, seed)
        _cache[key] = (w, te.upload_weights(w), {})
    w, dev, encs = _cache[key]
    if n_layers not in encs:
        if n_layers is None:
            m, dw = model, dev
        else:
            m = prefix_model(model, n_layers)
            dw = dict(dev, layers=dev["layers"][:n_layers])
        encs[n_layers] = te.Encoder(m, dw)
    return w, encs[n_layers]


def prefix_model(model, n_layers):
    return dict(model, n_encoder_layers=n_layers, n_decision_layers=0)


def prefix_weights(w, n_layers):
    return dict(w, layers=w["layers"][:n_layers])


def run_gpu(enc, ids, lengths, graphs=True):
    torch = require_gpu()
    B, S = ids.shape
    enc.set_graphs(graphs)
    out = torch.empty((B, S, enc.model["hidden"]), dtype=torch.bfloat16, device="cuda")
    enc.run(ids, lengths, out)
    enc.check()
    return to_bits(out)


def valid_rows(a, lengths):
    return np.concatenate([np.asarray(a)[b, :L] for b, L in enumerate(lengths)]).astype(np.float64)


def report(name, got_bits, ref, lengths):
    g = valid_rows(bf16_bits_to_f32(got_bits), lengths)
    r = valid_rows(ref, lengths)
    e, mabs = nrms(g, r), float(np.max(np.abs(g - r)))
    print(f"\n[parity] {name}: nRMS={e:.3e} max_abs={mabs:.3e} "
          f"frac(|d|<=2e-3)={np.mean(np.abs(g - r) <= 2e-3):.4f} max|ref|={np.max(np.abs(r)):.3f}")
    assert np.all(np.isfinite(g)), name
    return e, mabs


def check_full_depth(name, got_bits, model, w, ids, lengths):
    """GPU vs the fp32 and fp64-summed oracles, gated on the oracle's own spread."""
    t0 = time.time()
    r32 = oracle.forward(model, w, ids, lengths)
    r64 = oracle.forward(model, w, ids, lengths, accum_f64=True)
    floor = nrms(valid_rows(r32, lengths), valid_rows(r64, lengths))
    floor_abs = float(np.max(np.abs(valid_rows(r32, lengths) - valid_rows(r64, lengths))))
    print(f"\n[oracle] {name}: {time.time() - t0:.1f}s; floor nRMS(f32, f64)={floor:.3e} "
          f"max_abs={floor_abs:.3e}")
    e32, _ = report(name + " vs fp32 oracle", got_bits, r32, lengths)
    e64, m64 = report(name + " vs fp64 oracle", got_bits, r64, lengths)
    assert e64 <= 1.5 * floor + 1e-4, (name, e64, floor)
    assert e32 <= 2.0 * floor + 1e-4, (name, e32, floor)
    # max-abs: twice the oracle pair's own, plus one BF16 step at the largest
    # reference magnitude (one more flip of the largest element)
    step = float(ulp_bf16(np.max(np.abs(valid_rows(r64, lengths)))))
    assert m64 <= 2.0 * floor_abs + step, (name, m64, floor_abs, step)


def test_reduced_1x48_matches_oracle():
    model, B, S, seed, lr = synth.WORKLOADS["reduced_1x48"]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    e, _ = report("reduced 1x48", run_gpu(enc, ids, lengths), oracle.forward(model, w, ids, lengths),
                  lengths)
    assert e <= NRMS_LIMIT


@pytest.mark.parametrize("name,depth", [(n, d) for n in ("full_1x48", "full_4x64", "full_16x512")
                                        for d in (1, 2, 3, 4)])
def test_depth_prefix_within_page_limit(name, depth):
    model, B, S, seed, lr = synth.WORKLOADS[name]
    w, enc = encoder_for(model, seed, depth)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    rows = np.arange(B)
    got = run_gpu(enc, ids, lengths)
    for b in rows:
        L = int(lengths[b])
        ref = oracle.forward(prefix_model(model, depth), prefix_weights(w, depth), ids[b:b + 1, :L],
                             lengths[b:b + 1])
        e, _ = report(f"{name} row {b} after {depth} layer(s)", got[b:b + 1, :L], ref, [L])
        assert e <= NRMS_LIMIT, (name, depth, b, e)


@pytest.mark.parametrize("name", ["full_1x48", "full_4x64"])
def test_full_depth_small(name):
    model, B, S, seed, lr = synth.WORKLOADS[name]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    got = run_gpu(enc, ids, lengths)
    check_full_depth(name, got, model, w, ids, lengths)
    np.testing.assert_array_equal(got, run_gpu(enc, ids, lengths, graphs=False))  # eager == graph


@pytest.mark.parametrize("name", ["full_1x464", "full_4x464", "full_16x512"])
def test_full_depth_large_every_row(name):
    # the GPU runs the whole batch in the benchmarked configuration; the oracle
    # recomputes every row alone, truncated to its length (valid tokens do not
    # depend on padding: pinned by the oracle's own invariant tests)
    model, B, S, seed, lr = synth.WORKLOADS[name]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    got = run_gpu(enc, ids, lengths)
    for b in range(B):
        L = int(lengths[b])
        check_full_depth(f"{name} row {b} (len {L})", got[b:b + 1, :L], model, w,
                         ids[b:b + 1, :L], lengths[b:b + 1])


def test_full_depth_maximum_shape():
    # the largest request the library takes: max_batch rows of max_seq tokens,
    # every token valid (8192 tokens, no padding to skip); the first and the
    # last row against the oracle, every element finite
    model = synth.FULL
    B, S, seed = model["max_batch"], model["max_seq"], 4
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed)
    assert int(lengths.sum()) == B * S
    got = run_gpu(enc, ids, lengths)
    assert np.all(np.isfinite(bf16_bits_to_f32(got)))
    for b in (0, B - 1):
        check_full_depth(f"max {B}x{S} row {b}", got[b:b + 1], model, w, ids[b:b + 1],
                         lengths[b:b + 1])


def test_invariants_bitwise():
    model, B, S, seed, lr = synth.WORKLOADS["full_4x64"]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    a = run_gpu(enc, ids, lengths)
    # repeat, and a reused workspace after a different input with no readback
    other = (ids * 3 + 1) % model["vocab"]
    torch = require_gpu()
    tmp = torch.empty((B, S, model["hidden"]), dtype=torch.bfloat16, device="cuda")
    enc.run(other, lengths, tmp)
    np.testing.assert_array_equal(a, run_gpu(enc, ids, lengths))
    # padded ids do not change valid tokens
    ids2 = ids.copy()
    for b in range(B):
        ids2[b, lengths[b]:] = (ids2[b, lengths[b]:] + 17) % model["vocab"]
    c = run_gpu(enc, ids2, lengths)
    for b in range(B):
        np.testing.assert_array_equal(a[b, :lengths[b]], c[b, :lengths[b]])
    # row order: reversing the rows reverses the outputs
    r = run_gpu(enc, ids[::-1].copy(), lengths[::-1].copy())
    for b in range(B):
        L = lengths[b]
        np.testing.assert_array_equal(a[b, :L], r[B - 1 - b, :L])


@pytest.mark.parametrize("B,S", [(1, 1), (1, 16), (1, 63), (1, 64), (1, 65), (2, 127), (2, 128),
                                 (1, 129), (16, 1), (1, 511), (1, 512), (16, 64)])
def test_shape_boundaries(B, S):
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    ids, lengths = synth.make_inputs(model, B, S, 11, (1, S) if B > 1 else None)
    got = run_gpu(enc, ids, lengths)
    ref = oracle.forward(model, w, ids, lengths)
    e, _ = report(f"reduced {B}x{S}", got, ref, lengths)
    assert e <= NRMS_LIMIT


def test_invalid_arguments_enqueue_nothing():
    torch = require_gpu()
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    out = torch.full((2, 8, model["hidden"]), 7.0, dtype=torch.bfloat16, device="cuda")
    ids, lengths = synth.make_inputs(model, 2, 8, 0)
    cases = []
    bad = ids.copy()
    bad[1, 3] = model["vocab"]
    cases.append((bad, lengths))
    cases.append((ids, np.array([8, 0], np.int32)))
    cases.append((ids, np.array([9, 8], np.int32)))
    for i, l in cases:
        with pytest.raises(te.LayaError) as ex:
            enc.run(i, l, out)
        assert ex.value.code == te.E_INVAL
    big = np.zeros((17, 8), np.int32)
    with pytest.raises(te.LayaError):
        enc.run(big, np.full(17, 8, np.int32), out)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    enc.check()   # the handle is still usable


def test_run_device_matches_run():
    torch = require_gpu()
    model, B, S, seed, lr = synth.WORKLOADS["full_4x64"]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    a = run_gpu(enc, ids, lengths)
    out = torch.empty((B, S, model["hidden"]), dtype=torch.bfloat16, device="cuda")
    enc.run_device(i32_dev(ids), i32_dev(lengths), out)
    enc.check()
    np.testing.assert_array_equal(a, to_bits(out))


def test_encoder_stack_state_before_the_decision_layers():
    # the hidden state after the last encoder layer (the pages' "encoder27"
    # comparison point, #66 "Starting evidence"): the 28-layer encoder alone,
    # no final norm, gated like the full stack on the oracle's own spread
    model, B, S, seed, lr = synth.WORKLOADS["full_1x48"]
    n = model["n_encoder_layers"]
    w, enc = encoder_for(model, seed, n)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    got = run_gpu(enc, ids, lengths)
    check_full_depth("full_1x48 encoder stack", got, prefix_model(model, n), prefix_weights(w, n),
                     ids, lengths)


def test_empty_batch_is_rejected():
    torch = require_gpu()
    model = synth.REDUCED
    _, enc = encoder_for(model, 0)
    ids = np.zeros((0, 8), np.int32)
    out = torch.empty((0, 8, model["hidden"]), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(te.LayaError) as ex:
        enc.run(ids, np.zeros(0, np.int32), out)
    assert ex.value.code == te.E_INVAL
    enc.check()


def test_failure_poisons_the_handle_and_enqueues_nothing():
    # a failed launch (injected on the host, no device fault) stops this
    # handle: the failing call and every later one report it, the output is
    # untouched ("Laya native CUDA worker", "Start and check")
    torch = require_gpu()
    model = synth.REDUCED
    _, base = encoder_for(model, 0)
    enc = te.Encoder(base.model, base._weights)
    ids, lengths = synth.make_inputs(model, 1, 16, 3)
    out = torch.full((1, 16, model["hidden"]), 7.0, dtype=torch.bfloat16, device="cuda")
    enc.run(ids, lengths, out)
    enc.check()
    out.fill_(7.0)
    enc.debug_fail_next_run()
    with pytest.raises(te.LayaError) as ex:
        enc.run(ids, lengths, out)
    assert ex.value.code == te.E_CUDA
    for call in (lambda: enc.run(ids, lengths, out), lambda: enc.check()):
        with pytest.raises(te.LayaError) as ex:
            call()
        assert ex.value.code == te.E_POISONED
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    enc.close()
    fresh = te.Encoder(base.model, base._weights)   # other handles are unaffected
    fresh.run(ids, lengths, out)
    fresh.check()
    fresh.close()


def test_device_wait_runs_out_returns_device_error_and_fresh_handle_works():
    # "Laya native CUDA worker", "Start and check": a native failure stops the
    # executor.  The first projection's first CTA withholds one pipeline
    # stage, so its MMA issuer's bounded wait runs out (limit 50 ms): the
    # kernels return, laya_enc_check reports LAYA_E_DEVICE and poisons the
    # handle; a fresh handle on the same device then runs and matches the
    # oracle.  No trap, fault or invalid access is involved.
    torch = require_gpu()
    model, B, S, seed, lr = synth.WORKLOADS["reduced_1x48"]
    w = synth.make_weights(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    dev = te.upload_weights(w)
    enc = te.Encoder(model, dev)
    out = torch.empty((B, S, model["hidden"]), dtype=torch.bfloat16, device="cuda")
    try:
        enc.debug_set_wait_limit_ns(50_000_000)
        enc.debug_withhold_next_run()
        t0 = time.time()
        enc.run(ids, lengths, out)
        with pytest.raises(te.LayaError) as ex:
            enc.check()
        assert ex.value.code == te.E_DEVICE, ex.value
        assert time.time() - t0 < 30.0
        with pytest.raises(te.LayaError) as ex:
            enc.run(ids, lengths, out)
        assert ex.value.code == te.E_POISONED
    finally:
        enc.close()
    fresh = te.Encoder(model, dev)
    try:
        got = run_gpu(fresh, ids, lengths)
        e, _ = report("reduced 1x48 after a device error on another handle", got,
                      oracle.forward(model, w, ids, lengths), lengths)
        assert e <= NRMS_LIMIT
        with pytest.raises(te.LayaError):
            fresh.debug_set_wait_limit_ns(10)        # below 1 ms
    finally:
        fresh.close()
