"""Seeded synthetic inputs for the GEMM workloads (shared by tests and bench).

This module holds no GEMM arithmetic: it only draws random numbers with
numpy's ``default_rng``, rounds them to the storage dtype with torch's
round-to-nearest-even conversions, and lays them out K-major or MN-major.
Both the CUDA path and the oracle consume what it returns; neither is
imported here.

Storage conventions: A K-major is M x K row-major, A MN-major is K x M
row-major; B K-major is N x K row-major, B MN-major is K x N row-major
(rows of a K-major operand enumerate M/N, rows of an MN-major one enumerate
K).  Scale factors are plain row-major e8m0 bytes, [M][ceil(K/32)] for A and
[N][ceil(K/32)] for B.  The 6- and 4-bit formats (E3M2, E2M3, E2M1) are drawn
as uniformly random codes and stored packed, element i of the array in bits
[b*i, b*(i+1)) of one little-endian bit string (b = 6 or 4; leading
dimensions still count elements).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = ("f16", "bf16", "tf32", "e4m3", "e5m2", "e3m2", "e2m3", "e2m1", "nvf4")
#: bits per element of the packed formats ("nvf4": E2M1 elements of the
#: NVFP4 format, whose scales are unsigned E4M3 per 16 K elements)
PACKED_BITS = {"e3m2": 6, "e2m3": 6, "e2m1": 4, "nvf4": 4}
#: block-scaled formats: one e8m0 scale per 32 K elements, or for "nvf4" one
#: unsigned E4M3 scale per 16
BLOCK_SCALED = ("e4m3", "e5m2", "e3m2", "e2m3", "e2m1", "nvf4")
SCALE_BLOCK = {"nvf4": 16}

_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "tf32": torch.float32,
          "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
_BITS = {"f16": torch.int16, "bf16": torch.int16, "tf32": torch.int32, "e4m3": torch.uint8, "e5m2": torch.uint8}
_NP_BITS = {"f16": np.uint16, "bf16": np.uint16, "tf32": np.uint32, "e4m3": np.uint8, "e5m2": np.uint8}


@dataclass
class Workload:
    """One GEMM problem: shapes, operand dtype/majors, value distribution."""
    name: str
    M: int
    N: int
    K: int
    dtype: str                 # operand storage dtype: one of DTYPES
    a_major: str = "k"         # "k" | "mn"
    b_major: str = "k"
    dist: str = "normal"       # "normal": N(0,1)/sqrt(K); "uniform": U[-1,1]; "normal1": N(0,1)
    acc: str = "f32"           # accumulator dtype: f32 | f16
    out: str = "bf16"          # output dtype: f32 | f16 | bf16
    cta_group: int = 1
    block_scaled: bool = False
    seed_base: int = 0
    extra: dict = field(default_factory=dict)


# The five problems the benchmark and parity tests are built around.
WORKLOADS = {
    "tile_f16_128x128x64": Workload("tile_f16_128x128x64", 128, 128, 64, "f16", "k", "k",
                                    "uniform", "f32", "f32", 1, False, 1),
    "bf16_4096_kmn_cta1": Workload("bf16_4096_kmn_cta1", 4096, 4096, 4096, "bf16", "k", "mn",
                                   "normal", "f32", "bf16", 1, False, 2),
    # the workload leaves the CTA group open: the library's choice (pairs)
    "tf32_2048x2048x8192": Workload("tf32_2048x2048x8192", 2048, 2048, 8192, "tf32", "k", "k",
                                    "uniform", "f32", "f32", 0, False, 3),
    "bf16_8192_cta2": Workload("bf16_8192_cta2", 8192, 8192, 8192, "bf16", "k", "k",
                               "normal", "f32", "bf16", 2, False, 4),
    "f16acc_8192_cta2": Workload("f16acc_8192_cta2", 8192, 8192, 8192, "f16", "k", "k",
                                 "normal", "f16", "f16", 2, False, 4),
    "mxf8_8192": Workload("mxf8_8192", 8192, 8192, 8192, "e4m3", "k", "k",
                          "normal1", "f32", "bf16", 2, True, 5),
    # Block-scaled FP6 / FP4 (the same MMA kind with 6- and 4-bit elements):
    # uniformly random element codes, scales as for MXFP8.
    "mxf6_e2m3_8192": Workload("mxf6_e2m3_8192", 8192, 8192, 8192, "e2m3", "k", "k",
                               "codes", "f32", "bf16", 2, True, 8),
    "mxf4_8192": Workload("mxf4_8192", 8192, 8192, 8192, "e2m1", "k", "k",
                          "codes", "f32", "bf16", 2, True, 9),
    "nvf4_8192": Workload("nvf4_8192", 8192, 8192, 8192, "nvf4", "k", "k",
                          "codes", "f32", "bf16", 2, True, 10),
    # Skinny (decode-like) shapes: a few rows of activations against an
    # 8192 x 8192 weight; bound by streaming B from HBM, reported in GB/s.
    "bf16_skinny_m16": Workload("bf16_skinny_m16", 16, 8192, 8192, "bf16", "k", "k",
                                "normal", "f32", "bf16", 1, False, 6, {"bound": "hbm"}),
    "bf16_skinny_m128": Workload("bf16_skinny_m128", 128, 8192, 8192, "bf16", "k", "k",
                                 "normal", "f32", "bf16", 1, False, 7, {"bound": "hbm"}),
    # Chained product E = round(A.B1).B2 with a 256-wide intermediate kept in
    # tensor memory: M = 2 x 152 x 128 rows (two row tiles per SM), N = N2.
    "chain_bf16_38912x256x4096": Workload("chain_bf16_38912x256x4096", 38912, 4096, 4096, "bf16", "k", "k",
                                          "normal", "f32", "bf16", 1, False, 11, {"chain_n1": 256}),
}


def make_chain_inputs(w: Workload) -> dict:
    """Storage bits of a chained workload: A [M][K], B1 [N1][K] and B2
    [N][N1], all K-major; N(0,1) scaled by 1/sqrt of each product's K.
    Seeds 1000+i (A), 2000+i (B1), 2500+i (B2)."""
    n1 = w.extra["chain_n1"]
    i = w.seed_base
    A = to_bits(draw((w.M, w.K), 1000 + i, w.dist, w.K), w.dtype)
    B1 = to_bits(draw((n1, w.K), 2000 + i, w.dist, w.K), w.dtype)
    B2 = to_bits(draw((w.N, n1), 2500 + i, w.dist, n1), w.dtype)
    return {"A": A, "B1": B1, "B2": B2, "M": w.M, "N1": n1, "N2": w.N, "K": w.K}


def draw(shape, seed: int, dist: str, K: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist == "normal":
        return rng.standard_normal(size=shape) / np.sqrt(max(K, 1))
    if dist == "normal1":
        return rng.standard_normal(size=shape)
    if dist == "int4":  # small integers / 4 in [-1, 1]; exact sums
        return rng.integers(-4, 5, size=shape) / 4.0
    raise ValueError(dist)


def to_bits(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to the storage dtype (torch RNE) and return the raw
    storage bits as a numpy unsigned array."""
    t = torch.from_numpy(np.ascontiguousarray(x64, dtype=np.float64))
    if dtype in ("f16", "bf16", "e4m3", "e5m2"):
        t = t.to(torch.float32)  # exact for the draws used; then one RNE rounding
    t = t.to(_TORCH[dtype]).contiguous()
    return t.view(_BITS[dtype]).numpy().view(_NP_BITS[dtype]).copy()


def codes(shape, seed: int, bits: int) -> np.ndarray:
    """Uniformly random element codes of a `bits`-bit format."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << bits, size=shape, dtype=np.uint64).astype(np.uint8)


def pack(c: np.ndarray, bits: int) -> np.ndarray:
    """Pack a 2-D array of codes row by row into bytes: element j of a row in
    bits [bits*j, bits*(j+1)) of the row's little-endian bit string.  The row
    length times `bits` must be a multiple of 8."""
    rows, n = c.shape
    if (n * bits) % 8:
        raise ValueError("rows must fill whole bytes")
    v = c.astype(np.uint32)
    if bits == 4:
        out = v[:, 0::2] | (v[:, 1::2] << 4)
        return out.astype(np.uint8)
    if bits == 6:
        g = v.reshape(rows, n // 4, 4)
        word = g[..., 0] | (g[..., 1] << 6) | (g[..., 2] << 12) | (g[..., 3] << 18)
        out = np.stack([word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF], axis=-1)
        return out.reshape(rows, n // 4 * 3).astype(np.uint8)
    raise ValueError(bits)


def lay_out_a(a_logical: np.ndarray, major: str) -> np.ndarray:
    """Logical A (M x K) to storage (M x K for K-major, K x M for MN-major)."""
    return np.ascontiguousarray(a_logical if major == "k" else a_logical.T)


def lay_out_b(b_logical: np.ndarray, major: str) -> np.ndarray:
    """Logical B (K x N) to storage (N x K for K-major, K x N for MN-major)."""
    return np.ascontiguousarray(b_logical.T if major == "k" else b_logical)


def scales(rows: int, K: int, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """e8m0 scale bytes 127 + U{lo..hi}, one per 32 K elements per row."""
    rng = np.random.default_rng(seed)
    return (127 + rng.integers(lo, hi + 1, size=(rows, -(-K // 32)))).astype(np.uint8)


def ue4m3_scales(rows: int, K: int, seed: int) -> np.ndarray:
    """Unsigned E4M3 scale bytes, one per 16 K elements per row: exponent
    field uniform in 3..11 (2^-4 .. 2^4) and a uniform 3-bit fraction."""
    rng = np.random.default_rng(seed)
    shape = (rows, -(-K // 16))
    e = rng.integers(3, 12, size=shape)
    f = rng.integers(0, 8, size=shape)
    return ((e << 3) | f).astype(np.uint8)


def make_inputs(w: Workload, M: int | None = None, N: int | None = None, K: int | None = None,
                dist: str | None = None):
    """Storage-bit arrays (A, B, SFA, SFB) for a workload, optionally resized.

    Seeds follow the workload index: A 1000+i, B 2000+i, scales 3000+i (A) and
    4000+i (B).  Returns a dict with numpy arrays and leading dimensions.
    """
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    dist = w.dist if dist is None else dist
    i = w.seed_base
    if w.dtype in PACKED_BITS:
        # packed formats: K-major only; codes drawn per storage row
        if w.a_major != "k" or w.b_major != "k":
            raise ValueError("packed formats are stored K-major")
        bits = PACKED_BITS[w.dtype]
        A = pack(codes((M, K), 1000 + i, bits), bits)
        B = pack(codes((N, K), 2000 + i, bits), bits)
        out = {"A": A, "B": B, "lda": K, "ldb": K, "M": M, "N": N, "K": K, "SFA": None, "SFB": None}
    else:
        a = draw((M, K), 1000 + i, dist, K)
        b = draw((K, N), 2000 + i, dist, K)
        A = lay_out_a(to_bits(a, w.dtype), w.a_major)
        B = lay_out_b(to_bits(b, w.dtype), w.b_major)
        out = {"A": A, "B": B, "lda": A.shape[1], "ldb": B.shape[1], "M": M, "N": N, "K": K,
               "SFA": None, "SFB": None}
    if w.block_scaled and w.dtype == "nvf4":
        out["SFA"] = ue4m3_scales(M, K, 3000 + i)
        out["SFB"] = ue4m3_scales(N, K, 4000 + i)
    elif w.block_scaled:
        out["SFA"] = scales(M, K, 3000 + i)
        out["SFB"] = scales(N, K, 4000 + i)
    return out
