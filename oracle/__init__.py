"""Float64 CPU oracle for the tcgen05 swizzled GEMM and its layout probes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library never links, loads or calls it, and it shares no code with the
CUDA path.

* :func:`gemm` -- D = A.B (optionally block-scaled) and the error scale
  S = sum |a||b| in float64, from the raw storage bits (C, ``gemm_oracle.c``):
  fp32, f16, bf16, E4M3, E5M2, and the packed microscaling formats E3M2 /
  E2M3 (6 bits) and E2M1 (4 bits).
* :func:`gemm_chain` -- E = round(A.B1).B2, the product through a 16-bit
  intermediate, as two :func:`gemm` calls around :func:`encode_rne`.
* :mod:`oracle.layouts` -- the pages' descriptor walk, swizzles, TMEM
  register images, ldmatrix ownership and scale-factor placement.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against library routines, closed forms and the pages' worked examples.  Two
properties of the hardware are not modelled and stay "parity unpinned" (bounded
by the tolerance only): how the tensor cores round float32 storage to TF32
(the oracle reads the float32 values exactly; the per-product relative error
is at most 2^-10), and the order and rounding of fp16 accumulation inside the
MMA (the oracle accumulates in float64).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import layouts  # noqa: F401
from .build import LIB, build

F32, F16, BF16, E4M3, E5M2, E3M2, E2M3, E2M1 = 0, 1, 2, 3, 4, 5, 6, 7
#: bits per element of the packed formats (stored as a little-endian bit string)
PACKED_BITS = {E3M2: 6, E2M3: 6, E2M1: 4}
K_MAJOR, MN_MAJOR = 0, 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = LIB if os.path.exists(LIB) else build()
        lib = ctypes.CDLL(path)
        i64, vp, ci, dp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        lib.oracle_gemm.argtypes = [i64, i64, i64, vp, ci, ci, i64, vp, ci, ci, i64,
                                    vp, i64, vp, i64, ci, ci, vp, i64, dp, dp, ci]
        lib.oracle_gemm.restype = ci
        for name, t in (("oracle_dec_f16", ctypes.c_uint16), ("oracle_dec_bf16", ctypes.c_uint16),
                        ("oracle_dec_f32", ctypes.c_uint32), ("oracle_dec_e4m3", ctypes.c_uint8),
                        ("oracle_dec_e5m2", ctypes.c_uint8), ("oracle_dec_e3m2", ctypes.c_uint8),
                        ("oracle_dec_e2m3", ctypes.c_uint8), ("oracle_dec_e2m1", ctypes.c_uint8),
                        ("oracle_dec_e8m0", ctypes.c_uint8), ("oracle_dec_ue4m3", ctypes.c_uint8)):
            f = getattr(lib, name)
            f.argtypes = [t]
            f.restype = ctypes.c_double
        lib.oracle_num_threads.restype = ci
        _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Decode raw storage bits to float64 with the oracle's C decoders
    (element by element; meant for pins and small arrays)."""
    lib = _load()
    f = {F32: lib.oracle_dec_f32, F16: lib.oracle_dec_f16, BF16: lib.oracle_dec_bf16,
         E4M3: lib.oracle_dec_e4m3, E5M2: lib.oracle_dec_e5m2, E3M2: lib.oracle_dec_e3m2,
         E2M3: lib.oracle_dec_e2m3, E2M1: lib.oracle_dec_e2m1}[dtype]
    flat = np.asarray(bits).ravel()
    return np.array([f(int(x)) for x in flat], dtype=np.float64).reshape(np.shape(bits))


def decode_ue4m3(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits).ravel()
    return np.array([lib.oracle_dec_ue4m3(int(x)) for x in flat], dtype=np.float64).reshape(np.shape(bits))


#: scale encodings
SF_E8M0, SF_UE4M3 = 0, 1


def decode_e8m0(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits).ravel()
    return np.array([lib.oracle_dec_e8m0(int(x)) for x in flat],
                    dtype=np.float64).reshape(np.shape(bits))


_STORAGE = {F32: np.uint32, F16: np.uint16, BF16: np.uint16, E4M3: np.uint8, E5M2: np.uint8, E3M2: np.uint8,
            E2M3: np.uint8, E2M1: np.uint8}


def gemm(M: int, N: int, K: int, A: np.ndarray, a_type: int, a_major: int, lda: int,
         B: np.ndarray, b_type: int, b_major: int, ldb: int,
         SFA: np.ndarray | None = None, SFB: np.ndarray | None = None,
         rows=None, nthreads: int = 0, sf_block: int = 32, sf_kind: int = 0):
    """Float64 D and S for the requested rows (all rows when ``rows`` is None).

    A/B are raw storage arrays (uint32 for fp32, uint16 for f16/bf16, uint8 for
    e4m3 / e5m2, and uint8 bytes of the packed bit string for the 6- and 4-bit
    formats, whose ld is still counted in elements) laid out as the C file's
    header states.  SFA/SFB are plain
    row-major scale arrays [M][ceil(K/sf_block)] / [N][ceil(K/sf_block)]:
    e8m0 (sf_kind SF_E8M0, blocks of 32) or unsigned E4M3 (SF_UE4M3, the NVFP4
    blocks of 16).
    Returns (D, S) of shape (len(rows), N).
    """
    lib = _load()
    A = np.ascontiguousarray(A, dtype=_STORAGE[a_type])
    B = np.ascontiguousarray(B, dtype=_STORAGE[b_type])
    if rows is None:
        nrows = M
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        if nrows and (rows_arr.min() < 0 or rows_arr.max() >= M):
            raise ValueError("row index out of range")
    D = np.zeros((nrows, N), dtype=np.float64)
    S = np.zeros((nrows, N), dtype=np.float64)
    kb = -(-K // sf_block)
    sfa_p = sfb_p = None
    if SFA is not None:
        SFA = np.ascontiguousarray(SFA, dtype=np.uint8)
        assert SFA.shape == (M, kb), SFA.shape
        sfa_p = SFA.ctypes.data
    if SFB is not None:
        SFB = np.ascontiguousarray(SFB, dtype=np.uint8)
        assert SFB.shape == (N, kb), SFB.shape
        sfb_p = SFB.ctypes.data
    rc = lib.oracle_gemm(M, N, K, A.ctypes.data, a_type, a_major, lda,
                         B.ctypes.data, b_type, b_major, ldb,
                         sfa_p, kb, sfb_p, kb, sf_block, sf_kind,
                         None if rows_arr is None else rows_arr.ctypes.data, nrows,
                         D.ctypes.data, S.ctypes.data, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed with {rc}")
    return D, S


def encode_rne(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float64 values to f16 or bf16, nearest with ties to even, and
    return the storage bits (uint16).  f16 is numpy's correctly rounded
    float64 -> float16 conversion; bf16 (8 significant bits, exponent range
    of fp32) rounds x / q to an even integer with q the spacing of bf16
    numbers at |x| (2^(e-8) for |x| in [2^(e-1), 2^e), 2^-133 below the
    normal range), which is exact because q is a power of two; the result
    is an fp32 value whose upper 16 bits are the bf16 bits."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype != BF16:
        raise ValueError("encode_rne: f16 or bf16")
    _, e = np.frexp(x)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    y = np.rint(x / q) * q
    y = np.where(np.abs(y) > 3.3895313892515355e38, np.copysign(np.inf, x), y)
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gemm_chain(M: int, N1: int, N2: int, K: int, A: np.ndarray, B1: np.ndarray, B2: np.ndarray, dtype: int,
               lda: int = 0, ldb1: int = 0, ldb2: int = 0, rows=None):
    """E = round(A . B1) . B2 in float64 for the requested rows, with the
    intermediate C = A . B1 rounded to ``dtype`` (f16 / bf16) as a 16-bit
    intermediate would be; A [M][K], B1 [N1][K], B2 [N2][N1] are K-major
    storage bits.  Returns (E, S2, C, S1): S2 = sum |round(C)||B2| and
    S1 = sum |A||B1| are the error scales of the two products, C the exact
    float64 intermediate."""
    C, S1 = gemm(M, N1, K, A, dtype, K_MAJOR, lda or K, B1, dtype, K_MAJOR, ldb1 or K, rows=rows)
    Cbits = encode_rne(C, dtype)
    E, S2 = gemm(C.shape[0], N2, N1, Cbits, dtype, K_MAJOR, N1, B2, dtype, K_MAJOR, ldb2 or N1)
    return E, S2, C, S1
