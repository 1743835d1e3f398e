"""Python binding of the tcgen05 swizzled GEMM library (``include/tcg.h``).

Argument marshalling only: every function forwards to the C ABI of
``libtcg.so`` with the same name (``tcg_`` prefix dropped).  Tensors are
passed by ``data_ptr()``; streams default to torch's current CUDA stream.
No computation happens in Python and there is no fallback: if the library is
not built, every call raises ImportError.  Build it with
``python -c "import __graft_entry__ as g; g.build()"`` (or ``build.py``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtcg.so")

# enums (tcg.h)
OK, ERR_INVALID, ERR_ALIGNMENT, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_NO_DEVICE = 0, -1, -2, -3, -4, -5, -6
K_MAJOR, MN_MAJOR = 0, 1
F32, F16, BF16 = 0, 1, 2
IN_F16, IN_BF16, IN_TF32, IN_E4M3, IN_E5M2, IN_E3M2, IN_E2M3, IN_E2M1, IN_NVF4 = 0, 1, 2, 3, 4, 5, 6, 7, 8

_i64, _i32, _u32, _u64, _vp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_void_p


class GemmArgs(ctypes.Structure):
    """Mirror of ``tcg_gemm_args``."""
    _fields_ = [("M", _i64), ("N", _i64), ("K", _i64), ("in_type", _i32),
                ("A", _vp), ("a_major", _i32), ("lda", _i64),
                ("B", _vp), ("b_major", _i32), ("ldb", _i64),
                ("SFA", _vp), ("SFB", _vp), ("SFA_img", _vp), ("SFB_img", _vp),
                ("D", _vp), ("d_type", _i32), ("ldd", _i64), ("acc_type", _i32),
                ("cta_group", _i32), ("raster_group", _i32), ("sf_staging", _i32), ("split_k", _i32),
                ("epilogue", _i32)]


class ProbeOperand(ctypes.Structure):
    """Mirror of ``tcg_probe_operand``."""
    _fields_ = [("image", _vp), ("bytes", _i32), ("major", _i32), ("ldo", _u32), ("sdo", _u32),
                ("swizzle", _i32), ("start", _u32 * 8)]


_GEMM_SIG = [_i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _i32, _vp]
_SIGS = {
    "tcg_gemm_f16": (_GEMM_SIG, _i32),
    "tcg_gemm_bf16": (_GEMM_SIG, _i32),
    "tcg_gemm_tf32": (_GEMM_SIG, _i32),
    "tcg_gemm_mxf8_blockscaled": ([_i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i32,
                                   _i64, _i32, _vp], _i32),
    "tcg_gemm_mxf8_blockscaled_noalloc": ([_i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _vp,
                                           _i32, _i64, _i32, _vp], _i32),
    "tcg_gemm_mxf6_blockscaled": ([_i32, _i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i32,
                                   _i64, _i32, _vp], _i32),
    "tcg_gemm_mxf4_blockscaled": ([_i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i32,
                                   _i64, _i32, _vp], _i32),
    "tcg_gemm_nvf4_blockscaled": ([_i64, _i64, _i64, _vp, _i32, _i64, _vp, _i32, _i64, _vp, _vp, _vp, _i32,
                                   _i64, _i32, _vp], _i32),
    "tcg_scale_image_bytes": ([_i32, _i64, _i64, _i32], _i64),
    "tcg_prepare_scales_ab": ([_i32, _vp, _i64, _vp, _vp, _i64, _i32, _vp, _i64, _vp], _i32),
    "tcg_gemm": ([ctypes.POINTER(GemmArgs), _vp], _i32),
    "tcg_gemm_chain": ([_i32, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp, _i32, _i64, _vp], _i32),
    "tcg_mxf8_scale_image_bytes": ([_i64, _i64, _i32], _i64),
    "tcg_mxf8_tile_n": ([_i64, _i64, _i64, _i32, _i32], _i32),
    "tcg_tile_n": ([_i32, _i64, _i64, _i64, _i32, _i32], _i32),
    "tcg_mxf8_prepare_scales": ([_vp, _i64, _i64, _i32, _vp, _vp], _i32),
    "tcg_mxf8_prepare_scales_ab": ([_vp, _i64, _vp, _vp, _i64, _i32, _vp, _i64, _vp], _i32),
    "tcg_check": ([_vp], _i32),
    "tcg_set_wait_timeout_ns": ([_u64], None),
    "tcg_status_string": ([_i32], ctypes.c_char_p),
    "tcg_last_error_string": ([], ctypes.c_char_p),
    "tcg_last_launch_count": ([], _i32),
    "tcg_last_plan_string": ([], ctypes.c_char_p),
    "tcg_trace_next": ([_vp, _i32], _i32),
    "tcg_probe_tmem_roundtrip": ([_vp, _vp, _i32, _vp], _i32),
    "tcg_probe_cp": ([_vp, _i32, _i32, _u32, _u32, _u32, _i32, _vp, _vp], _i32),
    "tcg_probe_ld_shape": ([_vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_mma_tile": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_mma_tile_ws": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_mma_tmem_a": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_mma_ws64": ([_vp, _i32, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_mma_image": ([ctypes.POINTER(ProbeOperand), ctypes.POINTER(ProbeOperand), _i32, _i32, _i32, _vp,
                             _vp], _i32),
    "tcg_probe_ldmatrix_x2": ([_vp, _vp, _vp], _i32),
    "tcg_probe_stmatrix": ([_vp, _vp, _i32, _i32, _vp, _vp], _i32),
    "tcg_probe_ld_split": ([_vp, _i32, _i32, _i32, _vp, _vp, _vp], _i32),
    "tcg_probe_wait_timeout": ([_u64, _vp], _i32),
}

_lib_handle = None


def _load():
    """The loaded library; raises (never falls back) if it is not built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run blackwell_tensor_core_swizzled_gb300/build.py "
                              "(nvcc for sm_103a) first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib_handle = lib
    return _lib_handle


class _Lazy:
    def __getattr__(self, name):
        return getattr(_load(), name)


_lib = _Lazy()

EXPORTED = tuple(_SIGS)


class TcgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.tcg_status_string(status).decode()
        detail = _lib.tcg_last_error_string().decode()
        super().__init__(f"{where}: {msg} ({status})" + (f": {detail}" if detail else ""))


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ok(rc: int, where: str) -> int:
    if rc != 0:
        raise TcgError(rc, where)
    return rc


def gemm_f16(M, N, K, A, a_major, lda, B, b_major, ldb, D, d_type, ldd, acc_type=F32, stream=None):
    return _ok(_lib.tcg_gemm_f16(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(D), d_type, ldd,
                                 acc_type, _stream(stream)), "gemm_f16")


def gemm_bf16(M, N, K, A, a_major, lda, B, b_major, ldb, D, d_type, ldd, acc_type=F32, stream=None):
    return _ok(_lib.tcg_gemm_bf16(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(D), d_type, ldd,
                                  acc_type, _stream(stream)), "gemm_bf16")


def gemm_tf32(M, N, K, A, a_major, lda, B, b_major, ldb, D, d_type, ldd, acc_type=F32, stream=None):
    return _ok(_lib.tcg_gemm_tf32(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(D), d_type, ldd,
                                  acc_type, _stream(stream)), "gemm_tf32")


def gemm_mxf8_blockscaled(M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type=F32,
                          stream=None):
    return _ok(_lib.tcg_gemm_mxf8_blockscaled(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(SFA),
                                              _ptr(SFB), _ptr(D), d_type, ldd, acc_type, _stream(stream)),
               "gemm_mxf8_blockscaled")


def gemm_mxf6_blockscaled(fmt, M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type=F32,
                          stream=None):
    """Block-scaled FP6 GEMM (fmt IN_E3M2 or IN_E2M3; A and B packed, see tcg.h)."""
    return _ok(_lib.tcg_gemm_mxf6_blockscaled(fmt, M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(SFA),
                                              _ptr(SFB), _ptr(D), d_type, ldd, acc_type, _stream(stream)),
               "gemm_mxf6_blockscaled")


def gemm_mxf4_blockscaled(M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type=F32,
                          stream=None):
    """MXFP4 GEMM: packed E2M1, e8m0 scales per 32 K elements (see tcg.h)."""
    return _ok(_lib.tcg_gemm_mxf4_blockscaled(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(SFA),
                                              _ptr(SFB), _ptr(D), d_type, ldd, acc_type, _stream(stream)),
               "gemm_mxf4_blockscaled")


def gemm_nvf4_blockscaled(M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type=F32,
                          stream=None):
    """NVFP4 GEMM: packed E2M1, unsigned E4M3 scales per 16 K elements (see tcg.h)."""
    return _ok(_lib.tcg_gemm_nvf4_blockscaled(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(SFA),
                                              _ptr(SFB), _ptr(D), d_type, ldd, acc_type, _stream(stream)),
               "gemm_nvf4_blockscaled")


def scale_image_bytes(fmt, rows, K, tile_rows) -> int:
    return _lib.tcg_scale_image_bytes(fmt, rows, K, tile_rows)


def prepare_scales_ab(fmt, SFA, M, SFA_img, SFB, N, tile_n, SFB_img, K, stream=None):
    return _ok(_lib.tcg_prepare_scales_ab(fmt, _ptr(SFA), M, _ptr(SFA_img), _ptr(SFB), N, tile_n, _ptr(SFB_img), K,
                                          _stream(stream)), "prepare_scales_ab")


def gemm_mxf8_blockscaled_noalloc(M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd,
                                  acc_type=F32, stream=None):
    """The allocation-free MXFP8 GEMM (scale images in the library's fixed
    16 MiB device array; see include/tcg.h)."""
    return _ok(_lib.tcg_gemm_mxf8_blockscaled_noalloc(M, N, K, _ptr(A), a_major, lda, _ptr(B), b_major, ldb,
                                                      _ptr(SFA), _ptr(SFB), _ptr(D), d_type, ldd, acc_type,
                                                      _stream(stream)), "gemm_mxf8_blockscaled_noalloc")


def gemm_chain(in_type, M, N1, N2, K, A, lda, B1, ldb1, B2, ldb2, E, e_type, lde, stream=None, check=True):
    """Chained GEMM E = round(A . B1) . B2 with the intermediate in TMEM (``tcg_gemm_chain``)."""
    rc = _lib.tcg_gemm_chain(in_type, M, N1, N2, K, _ptr(A), lda, _ptr(B1), ldb1, _ptr(B2), ldb2, _ptr(E), e_type,
                             lde, _stream(stream))
    return _ok(rc, "gemm_chain") if check else rc


def gemm(M, N, K, in_type, A, a_major, lda, B, b_major, ldb, D, d_type, ldd, acc_type=F32, SFA=None, SFB=None,
         SFA_img=None, SFB_img=None, cta_group=0, raster_group=0, stream=None, check=True, sf_staging=0,
         split_k=0, epilogue=0):
    """Generic entry point (``tcg_gemm``); returns the status (raises if ``check``)."""
    a = GemmArgs(M, N, K, in_type, _ptr(A), a_major, lda, _ptr(B), b_major, ldb, _ptr(SFA), _ptr(SFB),
                 _ptr(SFA_img), _ptr(SFB_img), _ptr(D), d_type, ldd, acc_type, cta_group, raster_group,
                 sf_staging, split_k, epilogue)
    rc = _lib.tcg_gemm(ctypes.byref(a), _stream(stream))
    return _ok(rc, "gemm") if check else rc


def mxf8_scale_image_bytes(rows, K, tile_rows) -> int:
    return _lib.tcg_mxf8_scale_image_bytes(rows, K, tile_rows)


def mxf8_tile_n(M, N, K, b_major=K_MAJOR, cta_group=0) -> int:
    return _lib.tcg_mxf8_tile_n(M, N, K, b_major, cta_group)


def tile_n(fmt, M, N, K, b_major=K_MAJOR, cta_group=0) -> int:
    return _lib.tcg_tile_n(fmt, M, N, K, b_major, cta_group)


def mxf8_prepare_scales(sf, rows, K, tile_rows, img, stream=None):
    return _ok(_lib.tcg_mxf8_prepare_scales(_ptr(sf), rows, K, tile_rows, _ptr(img), _stream(stream)),
               "mxf8_prepare_scales")


def mxf8_prepare_scales_ab(SFA, M, SFA_img, SFB, N, tile_n, SFB_img, K, stream=None):
    return _ok(_lib.tcg_mxf8_prepare_scales_ab(_ptr(SFA), M, _ptr(SFA_img), _ptr(SFB), N, tile_n, _ptr(SFB_img), K,
                                               _stream(stream)), "mxf8_prepare_scales_ab")


def check(stream=None) -> int:
    """Synchronise the stream and return (not raise) the device error status."""
    return _lib.tcg_check(_stream(stream))


def set_wait_timeout_ns(ns: int) -> None:
    _lib.tcg_set_wait_timeout_ns(ns)


def status_string(status: int) -> str:
    return _lib.tcg_status_string(status).decode()


def last_error_string() -> str:
    return _lib.tcg_last_error_string().decode()


def last_launch_count() -> int:
    return _lib.tcg_last_launch_count()


def last_plan_string() -> str:
    return _lib.tcg_last_plan_string().decode()


def trace_next(buf, max_ctas: int):
    """Record the next GEMM launch's phase stamps into ``buf`` (see tcg.h)."""
    return _ok(_lib.tcg_trace_next(_ptr(buf), max_ctas), "trace_next")


def probe_tmem_roundtrip(inp, out, ncols, stream=None):
    return _ok(_lib.tcg_probe_tmem_roundtrip(_ptr(inp), _ptr(out), ncols, _stream(stream)), "probe_tmem_roundtrip")


def probe_cp(image, image_words, shape, origin_bytes, ldo, sdo, swizzle, out, stream=None):
    return _ok(_lib.tcg_probe_cp(_ptr(image), image_words, shape, origin_bytes, ldo, sdo, swizzle, _ptr(out),
                                 _stream(stream)), "probe_cp")


def probe_ld_shape(inp, shape, num, half, out, stream=None):
    return _ok(_lib.tcg_probe_ld_shape(_ptr(inp), shape, num, half, _ptr(out), _stream(stream)), "probe_ld_shape")


def probe_mma_tile(A, B, N, K, is_bf16, D, stream=None):
    return _ok(_lib.tcg_probe_mma_tile(_ptr(A), _ptr(B), N, K, is_bf16, _ptr(D), _stream(stream)), "probe_mma_tile")


def probe_mma_tile_ws(A, B, N, K, is_bf16, D, stream=None):
    return _ok(_lib.tcg_probe_mma_tile_ws(_ptr(A), _ptr(B), N, K, is_bf16, _ptr(D), _stream(stream)),
               "probe_mma_tile_ws")


def probe_mma_tmem_a(A, B, N, K, is_bf16, D, stream=None):
    return _ok(_lib.tcg_probe_mma_tmem_a(_ptr(A), _ptr(B), N, K, is_bf16, _ptr(D), _stream(stream)),
               "probe_mma_tmem_a")


def probe_mma_ws64(A, a_tmem, B, N, K, is_bf16, out, stream=None):
    return _ok(_lib.tcg_probe_mma_ws64(_ptr(A), a_tmem, _ptr(B), N, K, is_bf16, _ptr(out), _stream(stream)),
               "probe_mma_ws64")


def probe_operand(image, nbytes, major, ldo, sdo, swizzle, starts) -> ProbeOperand:
    st = (_u32 * 8)(*(list(starts) + [0] * (8 - len(starts))))
    return ProbeOperand(_ptr(image), nbytes, major, ldo, sdo, swizzle, st)


def probe_mma_image(a: ProbeOperand, b: ProbeOperand, in_type, N, ksteps, D, stream=None):
    return _ok(_lib.tcg_probe_mma_image(ctypes.byref(a), ctypes.byref(b), in_type, N, ksteps, _ptr(D),
                                        _stream(stream)), "probe_mma_image")


def probe_ldmatrix_x2(x, out, stream=None):
    return _ok(_lib.tcg_probe_ldmatrix_x2(_ptr(x), _ptr(out), _stream(stream)), "probe_ldmatrix_x2")


def probe_stmatrix(regs, row_off, count, trans, out, stream=None):
    return _ok(_lib.tcg_probe_stmatrix(_ptr(regs), _ptr(row_off), count, int(bool(trans)), _ptr(out),
                                       _stream(stream)), "probe_stmatrix")


def probe_ld_split(inp, num, imm_lanes, imm_cols, out_ld, out_st, stream=None):
    return _ok(_lib.tcg_probe_ld_split(_ptr(inp), num, imm_lanes, imm_cols, _ptr(out_ld), _ptr(out_st),
                                       _stream(stream)), "probe_ld_split")


def probe_wait_timeout(timeout_ns, stream=None):
    return _ok(_lib.tcg_probe_wait_timeout(timeout_ns, _stream(stream)), "probe_wait_timeout")


def raw_call(name: str, *args) -> int:
    """Call a C entry point by name with already-marshalled arguments (tests)."""
    return getattr(_lib, name)(*args)
