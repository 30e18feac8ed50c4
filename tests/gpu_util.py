"""Helpers shared by the GPU parity tests: device transfer of BF16 bit
patterns and the comparison measures (no arithmetic of the method)."""
import numpy as np

from transformer_encoder_bf16_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits


def require_gpu():
    import torch
    assert torch.cuda.is_available(), "GPU test run without a CUDA device"
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), f"expected a GB300 (10.3), got {major}.{minor}"
    return torch


def to_dev(bits, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(
        device).view(torch.bfloat16)


def to_bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def ulp_bf16(v):
    v = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(v)) - 7)


def nrms(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def bf16_close(got_bits, ref_bits, ulps=1.0, min_exact=0.95, rel_floor=2.0 ** -12):
    """Every element within `ulps` BF16 steps of the reference plus an absolute
    floor of rel_floor * max|ref|, and at least `min_exact` of them
    bit-identical.  The floor covers outputs that are small because their sum
    cancels: there the fp32 summation-order error is absolute (a fraction of
    the summed magnitudes), not relative to the result.  Returns (ok, message)."""
    g = bf16_bits_to_f32(got_bits).astype(np.float64)
    r = bf16_bits_to_f32(ref_bits).astype(np.float64)
    if not np.all(np.isfinite(g)):
        return False, "non-finite values"
    d = np.abs(g - r)
    floor = rel_floor * (float(np.max(np.abs(r))) if r.size else 0.0)
    lim = ulps * np.maximum(ulp_bf16(r), ulp_bf16(g)) + floor + 1e-30
    worst = float(np.max(d / lim)) if d.size else 0.0
    exact = float(np.mean(np.asarray(got_bits) == np.asarray(ref_bits))) if d.size else 1.0
    ok = worst <= 1.0 and exact >= min_exact
    return ok, f"worst {worst:.3f} of the allowed step, exact fraction {exact:.5f}"


def rnd_bits(rng, shape, std=1.0, mean=0.0):
    """Seeded normal draws rounded to BF16 bit patterns (test inputs)."""
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * std + mean)
