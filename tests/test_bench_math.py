"""The benchmark's own arithmetic, on CPU: algorithmic bytes and flops per
kernel class (the roofline numerators), the visible attention pairs, and the
rule that a recorded DRAM-traffic figure is dropped once the GEMM code
changes (comments alone do not count)."""
import os
import shutil
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from transformer_encoder_bf16_gb300 import synth  # noqa: E402

MODEL = synth.WORKLOADS["full_16x512"][0]


@pytest.mark.parametrize("M", [1, 48, 4117])
def test_projection_bytes_and_flops(M):
    H, I = MODEL["hidden"], MODEL["intermediate"]
    # weights once, activations in, outputs out (+ the residual read)
    assert bench.algorithmic(MODEL, "qkv", M) == (2 * (3 * H * H + M * H + M * 3 * H),
                                                  2.0 * M * 3 * H * H)
    assert bench.algorithmic(MODEL, "out_proj", M) == (2 * (H * H + M * H + 2 * M * H),
                                                       2.0 * M * H * H)
    assert bench.algorithmic(MODEL, "up_geglu", M) == (2 * (2 * I * H + M * H + M * I),
                                                       2.0 * M * 2 * I * H)
    assert bench.algorithmic(MODEL, "down", M) == (2 * (H * I + M * I + 2 * M * H),
                                                   2.0 * M * H * I)
    assert bench.algorithmic(MODEL, "norm", M) == (2 * (2 * M * H + H), 0.0)
    assert bench.algorithmic(MODEL, "rope", M) == (2 * 2 * 2 * M * H, 0.0)


def test_up_projection_flops_at_the_headline_size():
    # the per-launch figure the bench's roofline line reports at 16 x 512
    assert bench.algorithmic(MODEL, "up_geglu", 4117)[1] == 44249120768.0


@pytest.mark.parametrize("glob", [True, False])
def test_attention_pairs_match_brute_force(glob):
    rng = np.random.default_rng(5)
    lengths = rng.integers(1, 300, size=7)
    w = MODEL["local_half_window"]
    brute = 0
    for L in lengths:
        for i in range(L):
            for j in range(L):
                brute += 1 if (glob or abs(i - j) <= w) else 0
    assert bench.attention_pairs(MODEL, lengths, glob) == brute


def _copy_sources(dst):
    src = os.path.join(ROOT, "transformer_encoder_bf16_gb300", "csrc")
    os.makedirs(os.path.join(dst, "transformer_encoder_bf16_gb300", "csrc"))
    for name in bench.GEMM_SOURCES:
        shutil.copy(os.path.join(src, name), os.path.join(dst, "transformer_encoder_bf16_gb300",
                                                          "csrc", name))
    os.makedirs(os.path.join(dst, "profiles"))
    shutil.copy(os.path.join(ROOT, "profiles", "ncu_traffic.json"),
                os.path.join(dst, "profiles", "ncu_traffic.json"))


def test_traffic_record_follows_the_gemm_code(tmp_path, monkeypatch):
    _copy_sources(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    recorded = bench.recorded_traffic("full_16x512", "up_geglu")
    assert recorded is not None and recorded > 0   # the committed record matches the code
    gemm = tmp_path / "transformer_encoder_bf16_gb300" / "csrc" / "gemm.cu"
    text = gemm.read_text()
    gemm.write_text(text + "\n// a comment only\n\n")
    assert bench.recorded_traffic("full_16x512", "up_geglu") == recorded
    gemm.write_text(text + "\nstatic int changed_code = 1;\n")
    assert bench.recorded_traffic("full_16x512", "up_geglu") is None
    assert bench.recorded_traffic("full_16x512", "no_such_class") is None
