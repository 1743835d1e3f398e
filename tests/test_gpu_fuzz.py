"""Seeded random sweep of small problems through the C ABI, each compared in
full with the float64 oracle: operand dtype and majorness, ragged M / N / K
(including single rows, columns and K elements), CTA group, K decomposition
(library choice, one pass, stream-K, fixed split), output type and, for f16,
fp16 accumulation; a second sweep draws every block-scaled format (E4M3,
E5M2, E3M2, E2M3, E2M1 with e8m0 scales, NVFP4), the scale-staging mode and
the epilogue's drain shape.  Every case is reproducible from its index."""
import numpy as np
import pytest
import torch

import synthetic as syn
from gpu_helpers import TAU, assert_parity, make_case, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 80


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _draw(i):
    rng = np.random.default_rng(10_000 + i)
    dtype = ["f16", "bf16", "tf32", "e4m3"][rng.integers(4)]
    am, bm = ("k", "mn")[rng.integers(2)], ("k", "mn")[rng.integers(2)]
    def dim(hi):
        r = rng.random()
        return int(rng.integers(1, 33)) if r < 0.2 else int(rng.integers(1, hi + 1))
    M, N, K = dim(700), dim(700), dim(1200)
    cg = int(rng.integers(3))
    split = [0, 0, 1, -1, 3][rng.integers(5)]
    acc = "f16" if dtype == "f16" and rng.random() < 0.25 else "f32"
    out = "f16" if acc == "f16" else ["f32", "bf16", "f16"][rng.integers(3)]
    return dtype, am, bm, M, N, K, cg, split, acc, out


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_problem(tcg, oracle_mod, i):
    dtype, am, bm, M, N, K, cg, split, acc, out = _draw(i)
    x = make_case(dtype, am, bm, M, N, K, seed=20_000 + i)
    D = run_gpu(tcg, x, out=out, acc=acc, cta_group=cg, split_k=split)
    got = D[:M, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(got, ref, S, TAU[acc],
                  f"case {i}: {dtype} {am}{bm} {M}x{N}x{K} cg{cg} split {split} acc {acc} out {out} "
                  f"plan [{tcg.last_plan_string()}]", out)


N_SCALED = 48


def _draw_scaled(i):
    rng = np.random.default_rng(30_000 + i)
    dtype = ["e4m3", "e5m2", "e3m2", "e2m3", "e2m1", "nvf4"][rng.integers(6)]
    packed = dtype in syn.PACKED_BITS
    am = "k" if packed else ("k", "mn")[rng.integers(2)]
    bm = "k" if packed else ("k", "mn")[rng.integers(2)]
    def dim(hi):
        r = rng.random()
        return int(rng.integers(1, 33)) if r < 0.2 else int(rng.integers(1, hi + 1))
    M, N = dim(700), dim(1400)
    if dtype in ("e3m2", "e2m3"):
        K = 128 * int(rng.integers(1, 9))         # packed 6-bit rows: K a multiple of 128
    elif packed:
        K = 32 * int(rng.integers(1, 33))         # packed 4-bit rows: K a multiple of 32
    else:
        K = dim(1200)
    cg = int(rng.integers(3))
    split = [0, 0, 1, -1, 3][rng.integers(5)]
    staging = [0, 2][rng.integers(2)] if dtype in ("e2m1", "nvf4") else int(rng.integers(4))
    epilogue = int(rng.integers(3))
    # wide-range formats and raw codes can leave the f16 range: f32 / bf16 outputs there
    out = ["f32", "bf16", "f16"][rng.integers(3)] if dtype == "e4m3" else ["f32", "bf16"][rng.integers(2)]
    return dtype, am, bm, M, N, K, cg, split, staging, epilogue, out


@pytest.mark.parametrize("i", range(N_SCALED))
def test_random_block_scaled_problem(tcg, oracle_mod, i):
    dtype, am, bm, M, N, K, cg, split, staging, epilogue, out = _draw_scaled(i)
    dist = "codes" if dtype in syn.PACKED_BITS else "uniform"
    x = make_case(dtype, am, bm, M, N, K, dist=dist, seed=40_000 + i)
    D = run_gpu(tcg, x, out=out, cta_group=cg, split_k=split, sf_staging=staging, epilogue=epilogue)
    got = D[:M, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(got, ref, S, TAU["f32"],
                  f"case {i}: {dtype} {am}{bm} {M}x{N}x{K} cg{cg} split {split} staging {staging} "
                  f"epilogue {epilogue} out {out} plan [{tcg.last_plan_string()}]", out)
