"""The allocation-free MXFP8 entry point (tcg_gemm_mxf8_blockscaled_noalloc).

It is for callers that may not allocate device memory themselves or have the
library do it (a caching allocator that owns all device memory, or code that
cannot wait for the device-wide cudaFree of a growing workspace).  Its scale
images live in one fixed device array shared by all calls, so the test calls
it twice in a row, on different inputs, and checks each result against the
existing entry point's output for the same inputs.  This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TAU, assert_parity, make_case, oracle_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _run(fn, x, N):
    M, K = x["M"], x["K"]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn(M, N, K, to_device(x["A"]), 0, x["lda"], to_device(x["B"]), 0, x["ldb"], to_device(x["SFA"]),
       to_device(x["SFB"]), D, 2, N, 0)
    return D


def test_noalloc_matches_existing_entry_point_twice(tcg, oracle_mod):
    cases = [make_case("e4m3", "k", "k", 300, 520, 256, seed=31), make_case("e4m3", "k", "k", 1024, 1000, 512, seed=32)]
    results = []
    for x in cases:  # two calls in a row: the second reuses the shared array
        results.append(_run(tcg.gemm_mxf8_blockscaled_noalloc, x, x["N"]))
    assert tcg.check() == 0
    assert tcg.last_launch_count() == 3
    for x, got in zip(cases, results):
        ref_dev = _run(tcg.gemm_mxf8_blockscaled, x, x["N"])
        assert tcg.check() == 0
        _, S = oracle_rows(oracle_mod, x)
        assert_parity(got.double().cpu().numpy(), ref_dev.double().cpu().numpy(), S, TAU["f32"], "noalloc", "bf16")


def test_noalloc_rejects_problems_beyond_its_array(tcg):
    # 32768^3 needs far more than 16 MiB of scale images, whatever N tile is
    # chosen; the call must be rejected before anything is queued (the
    # pointers below are placeholders, so the precondition is checked first).
    n = 32768
    need = tcg.mxf8_scale_image_bytes(n, n, 128) + tcg.mxf8_scale_image_bytes(n, n, tcg.mxf8_tile_n(n, n, n))
    assert need > 2 * (16 << 20)
    rc = tcg.raw_call("tcg_gemm_mxf8_blockscaled_noalloc", n, n, n, 0x10000, 0, 0, 0x20000, 0, 0,
                      0x30000, 0x40000, 0x50000, 2, 0, 0, None)
    assert rc == tcg.ERR_UNSUPPORTED
    assert "16 MiB" in tcg.last_error_string()
