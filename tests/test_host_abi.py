"""Host-side checks of the C ABI (CPU only, no compute calls): the library
loads and exports every symbol the headers declare, configurations are
validated, the library's RoPE table equals the oracle's bit for bit, and the
GEMM planner keeps its invariants."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import transformer_encoder_bf16_gb300 as te
from transformer_encoder_bf16_gb300 import build as tebuild
from transformer_encoder_bf16_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    tebuild.build()
    return te.lib()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(laya_\w+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in te._SIGNATURES, f"binding lacks {n}"


def test_cache_stats_rejects_null_handle(lib):
    st = te.CacheStats()
    assert lib.laya_enc_get_cache_stats(None, ctypes.byref(st)) == te.E_INVAL
    assert ctypes.sizeof(te.CacheStats) == 2 * 4 + 6 * 8 + 2 * 8


def test_abi_version(lib):
    assert te.abi_version() == 3


def test_validate_config(lib):
    assert te.validate_config(synth.FULL) == te.OK
    assert te.validate_config(synth.REDUCED) == te.OK
    assert te.validate_config(dict(synth.FULL, out_fp32=1)) == te.OK
    for field, bad in (("hidden", 1000), ("head_dim", 32), ("heads", 15), ("intermediate", 2600),
                       ("max_seq", 513), ("max_batch", 17), ("global_every", 0),
                       ("local_half_window", -1), ("ln_eps", 0.0), ("vocab", 0),
                       ("n_encoder_layers", 0), ("final_norm", 2),
                       ("out_fp32", 2)):
        assert te.validate_config(dict(synth.FULL, **{field: bad})) == te.E_INVAL, field


@pytest.mark.parametrize("theta", [10000.0, 160000.0, 777.0])
@pytest.mark.parametrize("bf16", [True, False])
def test_rope_table_equals_oracle_bitwise(lib, orc, theta, bf16):
    c, s = te.rope_table(theta, 512, 32, bf16)
    oc, os_ = orc.rope_table(theta, 512, 32, bf16)
    np.testing.assert_array_equal(c.view(np.uint32), oc.view(np.uint32))
    np.testing.assert_array_equal(s.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M", [1, 7, 48, 100, 256, 257, 464, 1856, 8192])
@pytest.mark.parametrize("N,K,kind", [(3072, 1024, 0), (1024, 1024, 1), (2624, 1024, 2),
                                      (1024, 2624, 1), (768, 256, 0), (640, 256, 2),
                                      (2624, 1024, 3), (640, 256, 3)])
def test_linear_plan_invariants(lib, M, N, K, kind):
    for sms in (148, 152):
        nt, splits, ctas = te.linear_plan(M, K, N, kind, sms)
        assert nt % 16 == 0 and 16 <= nt <= 256
        tiles_t = -(-M // nt)
        assert tiles_t * nt >= M and (tiles_t - 1) * nt < M
        assert 1 <= splits <= min(16, K // 64)
        if kind == te.KIND_GEGLU_IL:
            assert splits == 1                         # interleaved GeGLU: unsplit plans only
        tiles = tiles_t * (N // 64 if kind == te.KIND_GEGLU_IL else -(-N // 128))
        if splits == 1:
            assert ctas == min(tiles, sms)             # persistent: one CTA per SM walks the tiles
        else:
            assert ctas == tiles * splits              # one CTA per (tile, split), clusters of `splits`
        if M <= 512 and K >= 1024 and kind != te.KIND_GEGLU_IL:
            # short sequences keep the GPU busy (the interleaved GeGLU has no
            # split-K: at a handful of tokens its 41 tiles are what it has, and
            # the forward's timing then picks the split two-tile GeGLU)
            assert ctas >= sms // 3


def test_linear_plan_rejects_bad_shapes(lib):
    with pytest.raises(te.LayaError):   # interleaved GeGLU needs N a multiple of 64
        te.linear_plan(48, 1024, 2600, te.KIND_GEGLU_IL, 152)
    with pytest.raises(te.LayaError):
        te.linear_plan(48, 100, 1024, 0, 148)      # K not a multiple of 64
    with pytest.raises(te.LayaError):
        te.linear_plan(0, 1024, 1024, 0, 148)


def test_create_reports_errors_without_a_gpu(lib):
    import ctypes
    import torch
    if torch.cuda.is_available():
        pytest.skip("host-only check")
    cfg = te.Config.from_model(synth.REDUCED)
    h = ctypes.c_void_p()
    # null weights: rejected before any CUDA call
    assert lib.laya_enc_create(ctypes.byref(cfg), None, ctypes.byref(h)) == te.E_INVAL
    assert not h.value
    assert lib.laya_enc_last_error(None)
    assert lib.laya_enc_destroy(None) == te.OK
    assert lib.laya_enc_run(None, None, None, 1, 1, None, None) == te.E_INVAL


def test_device_input_checks_reject_wrong_tensors():
    # host-side marshalling checks before the C ABI sees bare pointers (CPU
    # tensors stand for any tensor the checks must refuse)
    import torch
    ids = torch.zeros((2, 8), dtype=torch.int32)
    lens = torch.full((2,), 8, dtype=torch.int32)
    for a, b in ((ids, lens), (ids.long(), lens), (ids, lens.long()), (ids.t(), lens),
                 (ids, lens[:1]), (ids.reshape(-1), lens)):
        with pytest.raises(te.LayaError) as ex:
            te.check_device_inputs(a, b)
        assert ex.value.code == te.E_INVAL
