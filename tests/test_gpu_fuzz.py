"""Seeded random sweep of small problems through the C ABI, each compared in
full with the float64 oracle: operand dtype and majorness, ragged M / N / K
(including single rows, columns and K elements), CTA group, K decomposition
(library choice, one pass, stream-K, fixed split), output type and, for f16,
fp16 accumulation.  Every case is reproducible from its index."""
import numpy as np
import pytest
import torch

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
