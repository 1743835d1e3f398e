"""Helpers for the GPU parity tests: move storage-bit arrays to the device,
run the library through its C ABI, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import synthetic as syn

IN_TYPE = {"f16": 0, "bf16": 1, "tf32": 2, "e4m3": 3, "e5m2": 4, "e3m2": 5, "e2m3": 6, "e2m1": 7,
           "nvf4": 8}  # tcg_input
ORACLE_TYPE = {"f16": 1, "bf16": 2, "tf32": 0, "e4m3": 3, "e5m2": 4, "e3m2": 5, "e2m3": 6, "e2m1": 7,
               "nvf4": 7}  # oracle element enum (NVFP4 elements are E2M1)
ESIZE = {"f16": 2, "bf16": 2, "tf32": 4, "e4m3": 1, "e5m2": 1}   # bytes per element (unpacked formats)
OUT = {"f32": (0, torch.float32), "f16": (1, torch.float16), "bf16": (2, torch.bfloat16)}
ACC = {"f32": 0, "f16": 1}
TAU = {"f32": 2e-3, "f16": 1e-2}   # parity tolerance per accumulator type (x sum|a||b|)
# Unit roundoff of the output type: storing the fp32 accumulator as bf16/f16
# (round to nearest even) adds at most U_OUT * |D| on top of the accumulation
# error bounded by TAU * S.
U_OUT = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def to_device(bits: np.ndarray) -> torch.Tensor:
    view = {np.dtype(np.uint8): np.uint8, np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32}[bits.dtype]
    return torch.from_numpy(np.ascontiguousarray(bits).view(view)).cuda()


def pad_ld(bits: np.ndarray, esize: int, seed: int) -> np.ndarray:
    """Pad the rows of a storage array to a 16-byte multiple with random bits
    (which the GEMM must never read)."""
    rows, cols = bits.shape
    per = 16 // esize
    ld = max(per, -(-cols // per) * per)
    if ld == cols:
        return bits
    rng = np.random.default_rng(seed)
    out = rng.integers(0, np.iinfo(bits.dtype).max, size=(rows, ld), dtype=np.uint64).astype(bits.dtype)
    out[:, :cols] = bits
    return out


def make_case(dtype, am, bm, M, N, K, dist="uniform", seed=7, extra_pad=0):
    w = syn.Workload("case", M, N, K, dtype, am, bm, dist, block_scaled=(dtype in syn.BLOCK_SCALED), seed_base=seed)
    x = syn.make_inputs(w)
    x["w"] = w
    if dtype in syn.PACKED_BITS:  # packed rows of K elements (K a multiple of 128) are 32-byte multiples
        return x
    es = ESIZE[dtype]
    A = pad_ld(x["A"], es, seed + 11)
    B = pad_ld(x["B"], es, seed + 12)
    if extra_pad:
        per = 16 // es
        A = np.concatenate([A, np.zeros((A.shape[0], extra_pad * per), A.dtype)], axis=1)
        B = np.concatenate([B, np.zeros((B.shape[0], extra_pad * per), B.dtype)], axis=1)
    x["A"], x["B"], x["lda"], x["ldb"] = A, B, A.shape[1], B.shape[1]
    x["w"] = w
    return x


def run_gpu(tcg, x, out="bf16", acc="f32", cta_group=0, ldd=None, D=None, raster_group=0, sf_img=None, sf_staging=0,
            check=True, split_k=0, epilogue=0):
    w = x["w"]
    M, N, K = x["M"], x["N"], x["K"]
    dt, tdt = OUT[out]
    ldd = ldd or N
    A = to_device(x["A"])
    B = to_device(x["B"])
    if D is None:
        D = torch.full((max(M, 1), ldd), float("nan"), dtype=tdt, device="cuda")
    kw = {}
    if w.block_scaled:
        if sf_img is not None:
            kw = dict(SFA_img=sf_img[0], SFB_img=sf_img[1])
        else:
            kw = dict(SFA=to_device(x["SFA"]), SFB=to_device(x["SFB"]))
    tcg.gemm(M, N, K, IN_TYPE[w.dtype], A, 0 if w.a_major == "k" else 1, x["lda"], B,
             0 if w.b_major == "k" else 1, x["ldb"], D, dt, ldd, ACC[acc], cta_group=cta_group,
             raster_group=raster_group, sf_staging=sf_staging, split_k=split_k, epilogue=epilogue, **kw)
    if check:
        rc = tcg.check()
        assert rc == 0, f"{tcg.status_string(rc)}: {tcg.last_error_string()}"
    return D


def oracle_rows(oracle, x, rows=None):
    w = x["w"]
    t = ORACLE_TYPE[w.dtype]
    nv = w.dtype == "nvf4"  # unsigned E4M3 scales per 16 K elements
    return oracle.gemm(x["M"], x["N"], x["K"], x["A"], t, 0 if w.a_major == "k" else 1, x["lda"],
                       x["B"], t, 0 if w.b_major == "k" else 1, x["ldb"],
                       SFA=x["SFA"], SFB=x["SFB"], rows=rows, sf_block=16 if nv else 32,
                       sf_kind=oracle.SF_UE4M3 if nv else oracle.SF_E8M0)


def assert_parity(got: np.ndarray, ref: np.ndarray, S: np.ndarray, tau: float, what: str = "",
                  out: str = "f32"):
    """|got - ref| <= tau*S (accumulation) + u_out*(|ref| + tau*S) (output rounding).
    Returns max |got - ref| / S."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs at {np.argwhere(~np.isfinite(got))[:5]}"
    err = np.abs(got - ref)
    u = U_OUT[out]
    bad = err > tau * S + u * (np.abs(ref) + tau * S)
    if np.any(bad):
        idx = np.argwhere(bad)[:8]
        ratio = np.max(err / np.maximum(S, 1e-300))
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements beyond {tau}*S "
                             f"(max err/S {ratio:.3e}); first {idx.tolist()}: got "
                             f"{[float(got[tuple(i)]) for i in idx]} ref {[float(ref[tuple(i)]) for i in idx]}")
    return float(np.max(err / np.maximum(S, 1e-300))) if err.size else 0.0


def sample_rows(M: int, n: int = 12, seed: int = 0) -> list[int]:
    """Rows spread over tiles, TMEM lane quadrants and the ragged end."""
    base = {0, 1, 31, 32, 63, 64, 95, 96, 127, 128, 129, 255, 256, M // 2 + 77, M - 129, M - 2, M - 1}
    rng = np.random.default_rng(seed)
    base |= set(int(v) for v in rng.integers(0, M, size=n))
    return sorted(r for r in base if 0 <= r < M)
