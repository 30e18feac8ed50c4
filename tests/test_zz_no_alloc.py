"""laya_op_linear_noalloc: the projection for callers that cannot allocate
device memory (its split-K scratch is a fixed 16 MiB array inside the
library).  Checked through the C ABI against laya_op_linear, which takes a
caller workspace, on two calls in a row (the array keeps the previous call's
contents, which must not leak into the next).  This file is collected last."""
import numpy as np
import pytest

import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300.synth import f32_to_bf16_bits

from gpu_util import bf16_close, require_gpu, to_bits, to_dev

pytestmark = pytest.mark.gpu

MAX_SCRATCH = 16 << 20


def _bits(rng, shape, std=1.0):
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * std)


@pytest.mark.parametrize("kind,M,N,K,splits,nt", [
    (te.KIND_PLAIN, 48, 3072, 1024, 4, 48),     # split-K: scratch in use
    (te.KIND_GEGLU, 48, 2624, 1024, 6, 48),
    (te.KIND_RESIDUAL, 100, 1024, 2624, 7, 112),
    (te.KIND_PLAIN, 2000, 1024, 128, 1, 32),     # no split: no scratch needed
])
def test_noalloc_matches_linear_twice(kind, M, N, K, splits, nt):
    torch = require_gpu()
    assert te.linear_workspace_size(M, K, N, kind, splits, nt) <= MAX_SCRATCH
    rng = np.random.default_rng(M + N + K + kind)
    Nw = 2 * N if kind == te.KIND_GEGLU else N
    outs = []
    for call in range(2):
        x = to_dev(_bits(rng, (M, K)))
        w = to_dev(_bits(rng, (Nw, K), 0.02))
        r = to_dev(_bits(rng, (M, N))) if kind == te.KIND_RESIDUAL else None
        ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        te.linear(x, w, ref, kind, residual=r, splits=splits, tile_tokens=nt)
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        te.linear_noalloc(x, w, got, kind, residual=r, splits=splits, tile_tokens=nt)
        torch.cuda.synchronize()
        ok, msg = bf16_close(to_bits(got), to_bits(ref), ulps=1.0, min_exact=1.0)
        assert ok, (call, msg)                       # same kernel and plan: identical bytes
        outs.append(to_bits(got))
    assert not np.array_equal(outs[0], outs[1])      # the second call saw new inputs


def test_noalloc_rejects_plans_beyond_its_scratch():
    torch = require_gpu()
    M, N, K, splits, nt = 256, 2624, 1024, 4, 128   # 21 x 2 x 4 x 2 x 128 x 128 x 4 B = 22 MB of partials
    assert te.linear_workspace_size(M, K, N, te.KIND_GEGLU, splits, nt) > MAX_SCRATCH
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((2 * N, K), dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(te.LayaError) as ex:
        te.linear_noalloc(x, w, y, te.KIND_GEGLU, splits=splits, tile_tokens=nt)
    assert ex.value.code == te.E_INVAL
    torch.cuda.synchronize()
    assert torch.all(y == 3.0)                       # nothing was enqueued
