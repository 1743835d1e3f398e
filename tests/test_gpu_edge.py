"""Degenerate and extreme shapes through the C ABI against the float64 oracle.

Single elements, one-element K (less than one 128-byte K block: the rest of
the block is the TMA's zero fill), one row or one column in either
majorness, a very long K (2^19) whose one output tile is spread by stream-K
over every SM and summed from all their partial tiles, and a launch with
over a thousand tiles.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import TAU, assert_parity, make_case, oracle_rows, run_gpu, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


DEGENERATE = [
    # dtype, a_major, b_major, M, N, K, cta_group, out
    ("bf16", "k", "k", 1, 1, 1, 1, "f32"),
    ("f16", "mn", "mn", 1, 1, 1, 2, "f16"),
    ("tf32", "k", "mn", 1, 1, 1, 1, "f32"),
    ("e4m3", "k", "k", 1, 1, 1, 1, "bf16"),
    ("e4m3", "mn", "mn", 1, 1, 1, 2, "f32"),
    ("bf16", "k", "k", 300, 520, 1, 0, "bf16"),
    ("tf32", "mn", "k", 260, 300, 3, 2, "f32"),
    ("e4m3", "k", "mn", 200, 260, 16, 1, "bf16"),
    ("bf16", "k", "mn", 300, 1, 200, 1, "f32"),
    ("f16", "mn", "k", 1, 300, 200, 2, "f16"),
    ("bf16", "mn", "k", 513, 1, 72, 0, "bf16"),
    ("e4m3", "k", "k", 1, 257, 96, 0, "f32"),
    ("tf32", "k", "k", 129, 1, 40, 1, "bf16"),
]


@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out", DEGENERATE)
def test_degenerate_shapes_full_compare(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out):
    x = make_case(dtype, am, bm, M, N, K, seed=3 * M + 5 * N + K)
    D = run_gpu(tcg, x, out=out, acc="f32", cta_group=cg)
    got = D[:M, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(got, ref, S, TAU["f32"], f"{dtype} {am}{bm} {M}x{N}x{K}", out)


@pytest.mark.parametrize("split_k", [0, 5])
def test_very_long_k_stream_k(tcg, oracle_mod, split_k):
    # 128 x 136 x 2^19: one tile, 8192 K blocks; stream-K (default) spreads
    # them over every cluster, a fixed split of 5 gives uneven K ranges
    M, N, K = 128, 136, 1 << 19
    x = make_case("bf16", "k", "k", M, N, K, seed=17)
    D = run_gpu(tcg, x, out="f32", acc="f32", cta_group=1, split_k=split_k)
    plan = tcg.last_plan_string()
    assert ("stream-K" in plan) if split_k == 0 else ("split-K 5" in plan), plan
    rows = sample_rows(M, n=6)
    got = D[rows, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    assert_parity(got, ref, S, TAU["f32"], f"K=2^19 split {split_k}", "f32")


def test_many_tiles_one_launch(tcg, oracle_mod):
    # 65536 x 520 x 64: 512 M tiles x 3 N tiles (ragged), pairs
    M, N, K = 65536, 520, 64
    x = make_case("f16", "k", "k", M, N, K, seed=23)
    D = run_gpu(tcg, x, out="bf16", acc="f32", cta_group=2)
    rows = sample_rows(M, n=16)
    got = D[rows, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    assert_parity(got, ref, S, TAU["f32"], "65536x520x64", "bf16")
