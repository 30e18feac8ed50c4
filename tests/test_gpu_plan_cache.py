"""The projection plans chosen by timing, kept in a file across processes
(LAYA_PLAN_CACHE): a second process reads the first one's choices instead of
timing again, and runs exactly those plans."""
import json
import os
import subprocess
import sys

import pytest

from gpu_util import require_gpu

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, %r)
import torch
import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import synth
model, B, S, seed, lr = synth.WORKLOADS[sys.argv[1]]
enc = te.Encoder(model, te.upload_weights(synth.make_weights(model, seed)))
ids, lengths = synth.make_inputs(model, B, S, seed, lr)
out = torch.empty((B, S, model["hidden"]), dtype=torch.bfloat16, device="cuda")
enc.run(ids, lengths, out)
enc.check()
print(json.dumps({k: list(v) for k, v in enc.plans(B, S).items()}))
enc.close()
""" % ROOT


def _child(workload, cache):
    env = dict(os.environ, LAYA_PLAN_CACHE=cache)
    r = subprocess.run([sys.executable, "-c", CHILD, workload], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("workload", ["full_4x64", "full_16x512"])
def test_plan_cache_carries_plans_to_another_process(workload, tmp_path):
    require_gpu()
    cache = str(tmp_path / "plans.txt")
    first = _child(workload, cache)
    lines = open(cache).read().split("\n")
    rows = [ln.split() for ln in lines if ln.strip()]
    assert rows and all(len(r) == 9 for r in rows)
    # the second process reads the file and runs the same plans
    second = _child(workload, cache)
    assert second == first
