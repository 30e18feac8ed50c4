"""The fused short-request forward (one persistent kernel for batch * seq <=
128 tokens) against the CPU oracle and against the layer-by-layer kernels,
through the C ABI.

The two GPU paths compute the same layer equations with different split-K
boundaries, so they agree to rounding, not bitwise; each is held to the
oracle under the tolerance reading of test_gpu_forward.py (nRMS <= 5e-3 up to
four layers, the oracle's own fp32/fp64 spread at full depth).  What the
fused kernel must keep bitwise: repeated launches (its phase counters only
grow from one launch to the next), per-token independence (padding ids, row
order) and device-resident inputs."""
import numpy as np
import pytest

import oracle
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth

from gpu_util import i32_dev, require_gpu, to_bits
from test_gpu_forward import (NRMS_LIMIT, check_full_depth, encoder_for, prefix_model,
                              prefix_weights, report)

pytestmark = pytest.mark.gpu


def run(enc, ids, lengths, fused):
    torch = require_gpu()
    B, S = ids.shape
    enc.set_fused(fused)
    out = torch.empty((B, S, enc.model["hidden"]), dtype=torch.bfloat16, device="cuda")
    enc.run(ids, lengths, out)
    enc.check()
    return to_bits(out)


@pytest.mark.parametrize("B,S,lr", [(1, 1, None), (1, 16, None), (1, 48, None), (2, 40, (1, 40)),
                                    (4, 32, (5, 32)), (8, 16, (1, 16)), (1, 128, None),
                                    (16, 8, (1, 8)), (3, 33, (1, 33))])
def test_fused_reduced_matches_oracle(B, S, lr):
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    ids, lengths = synth.make_inputs(model, B, S, 5, lr)
    enc.set_fused(True)
    assert enc.launch_count(B, S) == 1
    ref = oracle.forward(model, w, ids, lengths)
    got = run(enc, ids, lengths, True)
    e, _ = report(f"fused reduced {B}x{S}", got, ref, lengths)
    assert e <= NRMS_LIMIT
    e2, _ = report(f"layered reduced {B}x{S}", run(enc, ids, lengths, False), ref, lengths)
    assert e2 <= NRMS_LIMIT


@pytest.mark.parametrize("depth", [1, 2, 3, 4])
@pytest.mark.parametrize("name,B,S,lr", [("full_1x48", 1, 48, None), ("full_2x64", 2, 64, (16, 64))])
def test_fused_depth_prefix_within_page_limit(name, B, S, lr, depth):
    model = synth.FULL
    w, enc = encoder_for(model, 1, depth)
    ids, lengths = synth.make_inputs(model, B, S, 1, lr)
    got = run(enc, ids, lengths, True)
    for b in range(B):
        L = int(lengths[b])
        ref = oracle.forward(prefix_model(model, depth), prefix_weights(w, depth), ids[b:b + 1, :L],
                             lengths[b:b + 1])
        e, _ = report(f"fused {name} row {b} after {depth} layer(s)", got[b:b + 1, :L], ref, [L])
        assert e <= NRMS_LIMIT, (name, depth, b, e)


def test_fused_full_depth_1x48():
    model, B, S, seed, lr = synth.WORKLOADS["full_1x48"]
    w, enc = encoder_for(model, seed)
    ids, lengths = synth.make_inputs(model, B, S, seed, lr)
    enc.set_fused(True)
    assert enc.launch_count(B, S) == 1
    got = run(enc, ids, lengths, True)
    check_full_depth("fused full_1x48", got, model, w, ids, lengths)
    layered = run(enc, ids, lengths, False)
    check_full_depth("layered full_1x48", layered, model, w, ids, lengths)


def test_fused_repeat_and_interleaved_shapes_bitwise():
    torch = require_gpu()
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    ids_a, len_a = synth.make_inputs(model, 2, 48, 7, (10, 48))
    ids_b, len_b = synth.make_inputs(model, 1, 96, 8, None)
    a0 = run(enc, ids_a, len_a, True)
    b0 = run(enc, ids_b, len_b, True)
    # many launches of two shapes (two workspaces, two counter sets), no sync between
    outs = []
    for i in range(6):
        ids, lens = (ids_a, len_a) if i % 2 == 0 else (ids_b, len_b)
        o = torch.empty((ids.shape[0], ids.shape[1], model["hidden"]), dtype=torch.bfloat16,
                        device="cuda")
        enc.run(ids, lens, o)
        outs.append(o)
    enc.check()
    for i, o in enumerate(outs):
        np.testing.assert_array_equal(to_bits(o), a0 if i % 2 == 0 else b0)


def test_fused_per_token_invariants_bitwise():
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    B, S = 4, 32
    ids, lengths = synth.make_inputs(model, B, S, 9, (3, 32))
    a = run(enc, ids, lengths, True)
    ids2 = ids.copy()
    for b in range(B):
        ids2[b, lengths[b]:] = (ids2[b, lengths[b]:] + 17) % model["vocab"]
    c = run(enc, ids2, lengths, True)
    for b in range(B):
        np.testing.assert_array_equal(a[b, :lengths[b]], c[b, :lengths[b]])
    r = run(enc, ids[::-1].copy(), lengths[::-1].copy(), True)
    for b in range(B):
        L = lengths[b]
        np.testing.assert_array_equal(a[b, :L], r[B - 1 - b, :L])


def test_fused_run_device_and_launch_counts():
    torch = require_gpu()
    model = synth.REDUCED
    w, enc = encoder_for(model, 0)
    ids, lengths = synth.make_inputs(model, 4, 32, 3, (1, 32))
    a = run(enc, ids, lengths, True)   # leaves the handle in fused mode
    out = torch.empty((4, 32, model["hidden"]), dtype=torch.bfloat16, device="cuda")
    enc.run_device(i32_dev(ids), i32_dev(lengths), out)
    enc.check()
    np.testing.assert_array_equal(a, to_bits(out))
    assert enc.launch_count(4, 32) == 1
    assert enc.launch_count(4, 33) > 1   # 132 tokens: the layer-by-layer kernels
    enc.set_fused(False)
    assert enc.launch_count(4, 32) > 1
    enc.set_fused(True)
