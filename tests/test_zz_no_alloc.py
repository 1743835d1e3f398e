"""The allocation-free MXFP8 entry point (tcg_gemm_mxf8_blockscaled_noalloc).

It is for callers that may not allocate device memory themselves or have the
library do it: a framework whose caching allocator owns all device memory, or
code that cannot wait for the device-wide cudaFree of a growing workspace.
Its scale images live in one fixed device array shared by all calls, so the
test calls it several times in a row -- a CTA-pair problem first, then
smaller ones that reuse the array over the first call's leftovers -- and
checks each result against the float64 oracle and, bit for bit, against the
allocating entry point (same kernel, same scale images).  A call on a stream
the library has never seen must not change the device's free memory, where
the allocating entry point would create a workspace.  This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TAU, assert_parity, make_case, oracle_rows, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _run(fn, x, stream=None):
    M, N, K = x["M"], x["N"], x["K"]
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fn(M, N, K, to_device(x["A"]), 0, x["lda"], to_device(x["B"]), 0, x["ldb"], to_device(x["SFA"]),
       to_device(x["SFB"]), D, 2, N, 0, stream=stream)
    return D


def test_noalloc_matches_oracle_and_existing_entry_point(tcg, oracle_mod):
    # large (CTA pairs: M > 128, N >= 1024) before small, so the later calls
    # read the shared array over the earlier calls' contents
    cases = [make_case("e4m3", "k", "k", 640, 1280, 512, seed=33),
             make_case("e4m3", "k", "k", 300, 520, 256, seed=31),
             make_case("e4m3", "k", "k", 130, 1024, 96, seed=34)]
    results, plans = [], []
    for x in cases:
        results.append(_run(tcg.gemm_mxf8_blockscaled_noalloc, x))
        plans.append(tcg.last_plan_string())
        assert tcg.last_launch_count() == 2  # both scale images in one launch, then the GEMM
    assert tcg.check() == 0
    assert plans[0].startswith("cta_group 2"), plans[0]
    assert plans[1].startswith("cta_group 1"), plans[1]
    for x, got in zip(cases, results):
        rows = sample_rows(x["M"], n=24, seed=x["M"]) if x["M"] > 400 else None
        ref, S = oracle_rows(oracle_mod, x, rows)
        g = got.double().cpu().numpy()
        if rows is not None:
            g = g[rows]
        assert_parity(g, ref, S, TAU["f32"], f"noalloc {x['M']}x{x['N']}x{x['K']}", "bf16")
        expected = _run(tcg.gemm_mxf8_blockscaled, x)
        assert tcg.check() == 0
        assert torch.equal(got.view(torch.int16), expected.view(torch.int16)), "differs from the allocating call"


def test_noalloc_allocates_nothing(tcg):
    # K = 32768 gives 4 MiB of scale images: the workspace the allocating
    # entry point creates for them is large enough to show in the device's
    # free memory (small allocations can come out of memory the driver holds
    # already).  The values do not matter here: bytes below 0x70 are finite
    # E4M3 numbers, and 127 is a scale of 1.
    M, N, K = 2048, 2048, 32768
    A = torch.randint(0, 0x70, (M, K), dtype=torch.uint8, device="cuda")
    B = torch.randint(0, 0x70, (N, K), dtype=torch.uint8, device="cuda")
    SFA = torch.full((M, K // 32), 127, dtype=torch.uint8, device="cuda")
    SFB = torch.full((N, K // 32), 127, dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert tcg.mxf8_scale_image_bytes(M, K, 128) + tcg.mxf8_scale_image_bytes(N, K, tcg.mxf8_tile_n(M, N, K)) \
        == 4 << 20

    def call(fn, stream):
        fn(M, N, K, A, 0, K, B, 0, K, SFA, SFB, D, 2, N, 0, stream=stream)

    s_warm, s_new, s_alloc = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    # load every kernel this uses (module loading may itself take memory)
    call(tcg.gemm_mxf8_blockscaled_noalloc, s_warm)
    assert tcg.check() == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    call(tcg.gemm_mxf8_blockscaled_noalloc, s_new)  # a stream the library has not seen
    assert tcg.check() == 0
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 >= free0, f"free device memory fell by {free0 - free1} bytes"
    # the allocating entry point on a fresh stream does create its workspace,
    # which the comparison above would have seen
    call(tcg.gemm_mxf8_blockscaled, s_alloc)
    assert tcg.check() == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] < free1


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


def test_noalloc_checks_every_argument_before_queueing(tcg):
    # invalid output type, ldd < N and a misaligned D fail on the host
    base = (256, 256, 64, 0x10000, 0, 0, 0x20000, 0, 0, 0x30000, 0x40000)
    assert tcg.raw_call("tcg_gemm_mxf8_blockscaled_noalloc", *base, 0x50000, 7, 0, 0, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_gemm_mxf8_blockscaled_noalloc", *base, 0x50000, 2, 100, 0, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_gemm_mxf8_blockscaled_noalloc", *base, 0x50001, 2, 0, 0, None) == tcg.ERR_ALIGNMENT
