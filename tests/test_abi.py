"""C-ABI checks that need no GPU: the library builds, loads, exports every
function ``include/tcg.h`` declares, and rejects bad arguments on the host
before touching the device.  Nothing here launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def tcg():
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "tcg.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tcg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_gemms():
    names = _declared()
    for n in ("tcg_gemm_f16", "tcg_gemm_bf16", "tcg_gemm_tf32", "tcg_gemm_mxf8_blockscaled"):
        assert n in names


def test_every_declared_symbol_is_exported(tcg):
    lib = ctypes.CDLL(tcg.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(tcg.EXPORTED) == _declared()


def test_status_strings(tcg):
    for s in range(0, -7, -1):
        assert tcg.status_string(s) != "unknown status"


def _call(tcg, name, M=256, N=256, K=64, A=0x10000, am=0, lda=0, B=0x20000, bm=0, ldb=0, D=0x30000,
          dt=2, ldd=0, acc=0):
    return tcg.raw_call(f"tcg_gemm_{name}", M, N, K, A, am, lda, B, bm, ldb, D, dt, ldd, acc, None)


def test_host_validation_rejects_bad_arguments(tcg):
    assert _call(tcg, "bf16", M=-1) == tcg.ERR_INVALID
    assert _call(tcg, "bf16", A=None) == tcg.ERR_INVALID
    assert _call(tcg, "bf16", D=None) == tcg.ERR_INVALID
    assert _call(tcg, "bf16", am=7) == tcg.ERR_INVALID
    assert _call(tcg, "bf16", lda=32) == tcg.ERR_INVALID            # lda < K
    assert _call(tcg, "bf16", ldd=100) == tcg.ERR_INVALID           # ldd < N
    assert _call(tcg, "bf16", A=0x10008) == tcg.ERR_ALIGNMENT       # TMA base alignment
    assert _call(tcg, "bf16", K=60, lda=60) == tcg.ERR_ALIGNMENT    # 120-byte rows
    assert _call(tcg, "bf16", acc=1, dt=1) == tcg.ERR_UNSUPPORTED   # bf16 with f16 accumulation
    assert _call(tcg, "f16", acc=1, dt=2) == tcg.ERR_UNSUPPORTED    # f16 accumulation needs f16 out
    assert _call(tcg, "tf32", dt=5) == tcg.ERR_INVALID
    # generic entry point: split_k below -1 (stream-K) is not a mode
    rc = tcg.gemm(256, 256, 64, 1, 0x10000, 0, 0, 0x20000, 0, 0, 0x30000, 2, 0, 0, split_k=-2, stream=0, check=False)
    assert rc == tcg.ERR_INVALID
    # mxf8 without scales
    rc = tcg.raw_call("tcg_gemm_mxf8_blockscaled", 64, 64, 64, 0x10000, 0, 0, 0x20000, 0, 0, None, None,
                      0x30000, 2, 0, 0, None)
    assert rc == tcg.ERR_INVALID
    # cp probe: shape codes 0..11 (4..11 decompressing), walk inside the image
    for shape in (-1, 12):
        assert tcg.raw_call("tcg_probe_cp", 0x10000, 512, shape, 0, 16, 128, 0, 0x20000, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_probe_cp", 0x10000, 256, 9, 0, 16, 128, 0, 0x20000, None) == tcg.ERR_INVALID
    # cp probe: a 4-row 4x256b walk whose 8-row blocks are not backed whole
    # (192 of the 256 bytes its two 16-byte columns organise) is rejected
    assert tcg.raw_call("tcg_probe_cp", 0x10000, 48, 3, 0, 128, 256, 0, 0x20000, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_probe_cp", 0x10000, 64, 3, 0, 128, 256, 0, 0x20000, None) != tcg.ERR_INVALID
    # MMA image probe: mode 4 is TF32 MN-major only, and a walk that could
    # leave its 96 KiB region under either stride assignment is rejected
    def op(major, sw, ldo, sdo, starts=(0,), nbytes=4096):
        return tcg.probe_operand(0x10000, nbytes, major, ldo, sdo, sw, starts)
    ok_a, ok_b = op(0, 3, 16, 1024), op(0, 3, 16, 1024)
    assert tcg.raw_call("tcg_probe_mma_image", ok_a, ok_b, 1, 64, 1, 0x30000, None) == tcg.ERR_NO_DEVICE
    assert tcg.raw_call("tcg_probe_mma_image", op(1, 4, 4096, 512), ok_b, 1, 64, 1, 0x30000,
                        None) == tcg.ERR_UNSUPPORTED
    assert tcg.raw_call("tcg_probe_mma_image", op(1, 3, 4096, 1024), ok_b, 2, 64, 1, 0x30000,
                        None) == tcg.ERR_UNSUPPORTED                                   # TF32 MN-major needs mode 4
    assert tcg.raw_call("tcg_probe_mma_image", op(1, 0, 128, 8192), ok_b, 1, 64, 1, 0x30000,
                        None) == tcg.ERR_INVALID                                       # 15 chunks x 8 KiB
    assert tcg.raw_call("tcg_probe_mma_image", op(0, 3, 16, 1024, starts=(8,)), ok_b, 1, 64, 1, 0x30000,
                        None) == tcg.ERR_INVALID                                       # origin not 16-byte aligned
    assert tcg.raw_call("tcg_probe_mma_image", ok_a, ok_b, 1, 72, 1, 0x30000, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_probe_mma_image", op(0, 3, 16, 1024, nbytes=200 * 1024), ok_b, 1, 64, 1, 0x30000,
                        None) == tcg.ERR_INVALID
    # trace request: buffer and count go together; null + 0 cancels
    assert tcg.raw_call("tcg_trace_next", None, 4) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_trace_next", 0x10000, 0) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_trace_next", 0x10004, 4) == tcg.ERR_ALIGNMENT
    assert tcg.raw_call("tcg_trace_next", None, 0) == tcg.OK
    # .ws probe: N must be one of the weight-stationary widths 64 / 128 / 256
    for n in (32, 96, 512):
        assert tcg.raw_call("tcg_probe_mma_tile_ws", 0x10000, 0x20000, n, 64, 0, 0x30000, None) == tcg.ERR_INVALID
    # split-access probe: repeat counts 1/2/4/8 and the four in-bounds immediates only
    for num, il, ic in ((3, 16, 8), (16, 16, 8), (4, 16, 4), (4, 0, 8), (4, 8, 0), (8, 32, 0)):
        assert tcg.raw_call("tcg_probe_ld_split", 0x10000, num, il, ic, 0x20000, 0x30000, None) == tcg.ERR_INVALID
    assert tcg.raw_call("tcg_probe_ld_split", None, 4, 16, 8, 0x20000, 0x30000, None) == tcg.ERR_INVALID
    # stmatrix probe: x1 / x2 / x4 only
    for count in (0, 3, 8):
        assert tcg.raw_call("tcg_probe_stmatrix", 0x10000, 0x20000, count, 0, 0x30000, None) == tcg.ERR_INVALID


def test_generic_entry_point_rejects_unknown_epilogue(tcg):
    for ep in (-1, 3):
        rc = tcg.gemm(256, 256, 64, tcg.IN_BF16, 0x10000, 0, 64, 0x20000, 0, 64, 0x30000, 2, 256,
                      check=False, epilogue=ep, stream=0)
        assert rc == tcg.ERR_INVALID


def test_chain_validation_before_any_device_work(tcg):
    # tcg_gemm_chain(in, M, N1, N2, K, A, lda, B1, ldb1, B2, ldb2, E, e_type, lde, stream)
    def call(in_type=1, M=64, N1=32, N2=64, K=64, A=0x10000, lda=64, B1=0x20000, ldb1=64, B2=0x30000, ldb2=32,
             E=0x40000, et=0, lde=64):
        return tcg.raw_call("tcg_gemm_chain", in_type, M, N1, N2, K, A, lda, B1, ldb1, B2, ldb2, E, et, lde, None)
    assert call(in_type=2) == tcg.ERR_INVALID                 # tf32: 16-bit operands only
    for n1 in (0, 8, 40, 272):
        assert call(N1=n1) == tcg.ERR_INVALID                 # N1 a multiple of 16 in [16, 256]
    assert call(M=-1) == tcg.ERR_INVALID
    assert call(et=5) == tcg.ERR_INVALID
    assert call(E=None) == tcg.ERR_INVALID
    assert call(lde=32) == tcg.ERR_INVALID                    # lde < N2
    assert call(E=0x40008) == tcg.ERR_ALIGNMENT               # E base
    assert call(et=2, lde=68) == tcg.ERR_ALIGNMENT            # 136-byte rows of E
    assert call(A=0x10008) == tcg.ERR_ALIGNMENT
    assert call(lda=60) == tcg.ERR_INVALID                    # lda < K
    assert call(ldb2=16) == tcg.ERR_INVALID                   # ldb2 < N1
    assert call(M=0, A=None, B1=None, B2=None, E=None) == tcg.OK
    assert call(N2=0, A=None, B1=None, B2=None, E=None) == tcg.OK


def test_empty_problems_are_noops(tcg):
    # M == 0 or N == 0 returns before any device work, even with null pointers
    assert _call(tcg, "bf16", M=0, A=None, B=None, D=None) == tcg.OK
    assert _call(tcg, "f16", N=0, A=None, B=None, D=None) == tcg.OK


def test_scale_image_sizes(tcg):
    # [K step][tile][chunk][512 B]: K=8192 -> 256 blocks -> 64 steps
    assert tcg.mxf8_scale_image_bytes(8192, 8192, 128) == 64 * 64 * 512
    assert tcg.mxf8_scale_image_bytes(8192, 8192, 224) == 64 * 37 * 2 * 512
    assert tcg.mxf8_scale_image_bytes(300, 96, 128) == 1 * 3 * 512
    assert tcg.mxf8_scale_image_bytes(8192, 8192, 256) == 64 * 32 * 2 * 512
    # N = 256 tiles for one CTA and for a pair (a pair's MN-major B half tile
    # is one whole 128-byte swizzle span of E4M3); pairs with K-major B over
    # at least 300 tiles of 256 x 384 take those
    for cg in (0, 1, 2):
        assert tcg.mxf8_tile_n(8192, 8192, 8192, tcg.K_MAJOR, cg) == 256
        assert tcg.mxf8_tile_n(8192, 8192, 8192, tcg.MN_MAJOR, cg) == 256
        for fmt in (tcg.IN_E5M2, tcg.IN_E3M2, tcg.IN_E2M3):
            assert tcg.tile_n(fmt, 8192, 8192, 8192, tcg.K_MAJOR, cg) == 256
        # packed FP4 pairs with K-major B over at least 300 tiles of 256 x 384
        for fmt in (tcg.IN_E2M1, tcg.IN_NVF4):
            assert tcg.tile_n(fmt, 8192, 8192, 8192, tcg.K_MAJOR, cg) == (256 if cg == 1 else 384)
    assert tcg.tile_n(tcg.IN_E2M1, 4096, 4096, 4096, tcg.K_MAJOR, 2) == 256      # 16 x 11 = 176 tiles
    assert tcg.tile_n(tcg.IN_NVF4, 2600, 10668, 256, tcg.K_MAJOR, 0) == 384      # 11 x 28 = 308
    assert tcg.tile_n(tcg.IN_BF16, 8192, 8192, 8192, tcg.K_MAJOR, 0) == tcg.ERR_INVALID
    assert tcg.scale_image_bytes(tcg.IN_E2M1, 8192, 8192, 384) == 32 * 22 * 3 * 2 * 512


@pytest.mark.skipif(os.environ.get("CUDA_VISIBLE_DEVICES_FORCE_GPU") is not None, reason="GPU present")
def test_fails_loudly_without_a_device(tcg):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call(tcg, "bf16") == tcg.ERR_NO_DEVICE
    with pytest.raises(tcg.TcgError):
        tcg.gemm_bf16(256, 256, 64, 0x10000, 0, 0, 0x20000, 0, 0, 0x30000, 2, 0, 0, stream=0)
