"""Operand images for the MMA image probe, laid out by the oracle's model of
the shared-descriptor walk ("tcgen05.mma" page, "Shared descriptors are
byte-stride contracts" and "swizzle=4").

Each case names, for A (128 x K) and B (N x K), the majorness, the pages'
swizzle mode and the two descriptor strides.  The MMA issues advance through
K in steps of 32 bytes (K = 16 for 16-bit inputs, 8 for TF32); where issue j
starts is the test's choice (as the GEMM's ring stages are), and the model
gives the walk from that origin:

    physical byte of element (mn, k) of issue j
        = swizzle(start_j + mma_operand_offset(mn, k - j*kstep))

The GPU probe copies the images into shared memory and lets the hardware walk
them; a mismatch with the oracle's GEMM of the logical operands means the
model (or the start rule) is wrong.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from oracle import layouts as L

ESIZE = {"f16": 2, "bf16": 2, "tf32": 4}


@dataclass(frozen=True)
class Spec:
    major: str      # "k" | "mn"
    swizzle: int    # the pages' logical mode 0..4
    ldo: int
    sdo: int


@dataclass(frozen=True)
class Case:
    name: str
    dtype: str
    N: int
    K: int
    a: Spec
    b: Spec


CASES = [
    Case("bf16 A K sw128, B MN sw128", "bf16", 128, 64, Spec("k", 3, 16, 1024), Spec("mn", 3, 8192, 1024)),
    Case("f16 A MN sw64, B K sw64", "f16", 64, 64, Spec("mn", 2, 4096, 512), Spec("k", 2, 16, 512)),
    Case("bf16 A MN sw32, B MN sw32", "bf16", 96, 32, Spec("mn", 1, 1024, 256), Spec("mn", 1, 1024, 256)),
    Case("f16 A MN none, B K none", "f16", 64, 64, Spec("mn", 0, 128, 1024), Spec("k", 0, 128, 1024)),
    Case("bf16 MN none, chunks first and gapped", "bf16", 32, 64, Spec("mn", 0, 2048, 128),
         Spec("mn", 0, 768, 128)),
    Case("tf32 A MN sw4, B MN sw4", "tf32", 64, 32, Spec("mn", 4, 4096, 512), Spec("mn", 4, 4096, 512)),
    Case("tf32 A K sw128, B K sw64", "tf32", 48, 32, Spec("k", 3, 16, 1024), Spec("k", 2, 16, 512)),
    Case("tf32 A K none, B MN sw4 N256", "tf32", 256, 16, Spec("k", 0, 2048, 128), Spec("mn", 4, 2048, 512)),
    Case("f16 A K sw32, B K sw128 N256", "f16", 256, 48, Spec("k", 1, 16, 256), Spec("k", 3, 16, 1024)),
    Case("bf16 A MN sw128, B MN sw64 N256", "bf16", 256, 64, Spec("mn", 3, 8192, 1024), Spec("mn", 2, 4096, 512)),
]


def kstep(dtype: str) -> int:
    """K elements per MMA issue: 32 bytes of K."""
    return 32 // ESIZE[dtype]


def issue_starts(spec: Spec, rows_mn: int, dtype: str, ksteps: int) -> list[int]:
    """Descriptor origin (bytes from the image start) of each MMA issue.

    K-major swizzled: issues advance 32 bytes along a row; once a row is used
    up the next K block is a separate tile of ceil(rows/8) row groups.
    K-major unswizzled: two 16-byte K chunks (LDO apart) per issue.
    MN-major: kstep K rows per issue, i.e. kstep/g row groups (g = 8, or 4
    for mode 4), SDO apart when swizzled and LDO apart when not.
    """
    es = ESIZE[dtype]
    ks = kstep(dtype)
    out = []
    for j in range(ksteps):
        if spec.major == "k":
            if spec.swizzle == 0:
                out.append(j * 2 * spec.ldo)
            else:
                per_row = L.row_bytes(spec.swizzle) // 32
                tile = -(-rows_mn // 8) * spec.sdo
                out.append((j // per_row) * tile + (j % per_row) * 32)
        else:
            g = L.rows_per_group(spec.swizzle)
            if spec.swizzle == 0:
                out.append(j * (ks // 8) * spec.ldo)
            else:
                out.append(j * (ks // g) * spec.sdo)
    del es
    return out


def element_addresses(spec: Spec, rows_mn: int, dtype: str, ksteps: int, starts=None, ldo=None, sdo=None):
    """Physical byte address of every element (mn, k), shape (rows_mn, K),
    under the oracle's model (optionally with other strides)."""
    es = ESIZE[dtype]
    ks = kstep(dtype)
    ldo = spec.ldo if ldo is None else ldo
    sdo = spec.sdo if sdo is None else sdo
    starts = issue_starts(spec, rows_mn, dtype, ksteps) if starts is None else starts
    mn = np.arange(rows_mn)[:, None]
    kk = np.arange(ks)[None, :]
    cols = []
    for j in range(ksteps):
        logical = starts[j] + L.mma_operand_offset(mn, kk, es, spec.major, ldo, sdo, spec.swizzle)
        cols.append(L.swizzle_addr(logical, spec.swizzle))
    return np.concatenate(cols, axis=1)


def build_image(bits: np.ndarray, spec: Spec, dtype: str, ksteps: int) -> np.ndarray:
    """The operand's shared bytes (uint8, a multiple of 16 long) with element
    (mn, k) of ``bits`` (rows_mn x K storage bits) at its modelled address;
    raises if two elements would share a byte."""
    es = ESIZE[dtype]
    rows_mn = bits.shape[0]
    addr = element_addresses(spec, rows_mn, dtype, ksteps)
    flat = addr.ravel()
    if np.unique(flat // es).size != flat.size:
        raise ValueError("two elements map to the same bytes")
    size = int(flat.max()) + es
    img = np.zeros(-(-size // 16) * 16, dtype=np.uint8)
    vals = bits.astype(np.uint64).ravel()
    for b in range(es):
        img[flat + b] = ((vals >> np.uint64(8 * b)) & np.uint64(0xFF)).astype(np.uint8)
    return img
