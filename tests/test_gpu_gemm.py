"""GEMM parity: the CUDA path through the C ABI against the float64 oracle.

Tolerance (per element): |D_gpu - D_ref| <= tau * sum_k |a||b| with tau = 2e-3
for fp32 accumulation and 1e-2 for fp16 accumulation.  Small cases compare
every element (several tiles, ragged tails in M, N and K); the full-size
workloads compare sampled rows (all N columns of each) in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import synthetic as syn
from gpu_helpers import IN_TYPE, TAU, assert_parity, make_case, oracle_rows, run_gpu, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _check_full(tcg, oracle_mod, x, out, acc, cg, **kw):
    D = run_gpu(tcg, x, out=out, acc=acc, cta_group=cg, **kw)
    got = D[:x["M"], :x["N"]].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x)
    return assert_parity(got, ref, S, TAU[acc], f"{x['w'].dtype} {x['w'].a_major}{x['w'].b_major} cg{cg}", out)


SMALL = [
    # dtype, a_major, b_major, M, N, K, cta_group, out, acc
    ("f16", "k", "k", 128, 128, 64, 1, "f32", "f32"),
    ("f16", "k", "k", 128, 128, 64, 2, "f32", "f32"),
    ("bf16", "k", "mn", 300, 520, 200, 1, "bf16", "f32"),
    ("bf16", "k", "k", 300, 520, 200, 2, "bf16", "f32"),
    ("bf16", "mn", "k", 513, 300, 136, 2, "f32", "f32"),
    ("bf16", "mn", "mn", 257, 257, 264, 1, "f16", "f32"),
    ("bf16", "k", "k", 1000, 1100, 640, 0, "bf16", "f32"),
    ("f16", "k", "k", 640, 768, 512, 2, "f16", "f16"),
    ("f16", "mn", "mn", 200, 300, 96, 1, "f16", "f16"),
    ("f16", "k", "mn", 384, 512, 1024, 1, "f16", "f16"),
    ("tf32", "k", "k", 300, 520, 200, 1, "f32", "f32"),
    ("tf32", "mn", "mn", 260, 300, 72, 2, "f32", "f32"),
    ("tf32", "k", "mn", 128, 256, 128, 1, "f32", "f32"),
    ("tf32", "mn", "k", 384, 256, 96, 2, "bf16", "f32"),
    # skinny variant (M <= 32, K-major A): 32 staged A rows, 64-wide tiles
    ("bf16", "k", "k", 20, 700, 1000, 1, "bf16", "f32"),
    ("bf16", "k", "k", 1, 300, 200, 0, "f32", "f32"),
    ("bf16", "k", "mn", 16, 520, 392, 1, "f16", "f32"),
    ("f16", "k", "mn", 32, 520, 640, 1, "f16", "f16"),
    # 33..64 and 65..128 rows: the same 64-wide tiles with 64 / 128 staged A rows
    ("bf16", "k", "k", 48, 700, 1000, 1, "bf16", "f32"),
    ("f16", "k", "mn", 64, 330, 264, 0, "f32", "f32"),
    ("bf16", "k", "k", 100, 520, 640, 0, "f16", "f32"),
    ("f16", "k", "k", 127, 300, 136, 1, "f16", "f16"),
    # narrow N (N <= 32, K-major B): 128 x 32 tiles
    ("bf16", "k", "k", 700, 20, 1000, 1, "bf16", "f32"),
    ("f16", "mn", "k", 300, 32, 72, 0, "f16", "f32"),
    ("f16", "k", "k", 300, 24, 136, 1, "f16", "f16"),     # f16 accumulation: packed TMEM loads
    ("e4m3", "k", "k", 300, 520, 256, 2, "bf16", "f32"),
    ("e4m3", "k", "k", 300, 520, 208, 1, "f32", "f32"),
    ("e4m3", "k", "k", 512, 448, 512, 2, "bf16", "f32"),
    ("e4m3", "mn", "mn", 200, 300, 256, 1, "bf16", "f32"),
    ("e4m3", "mn", "k", 260, 230, 160, 2, "f32", "f32"),
]


@pytest.mark.parametrize("split_k", [0, 1])
@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out,acc", SMALL)
def test_small_ragged_full_compare(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out, acc, split_k):
    # split_k 0: the library's choice (one pass for these); 1: one pass
    # per tile requested explicitly
    x = make_case(dtype, am, bm, M, N, K, seed=M + N + K)
    _check_full(tcg, oracle_mod, x, out, acc, cg, split_k=split_k)


# The block-scaled formats on kind::mxf8f6f4 besides E4M3: E5M2 bytes, and the
# packed FP6 (E3M2, E2M3) and FP4 (E2M1) formats, K-major and K a multiple of
# 128 for the packed ones; ragged M and N, single CTAs and pairs.
MX_FORMATS = [
    ("e5m2", "k", "k", 300, 520, 256, 2, "bf16"),
    ("e5m2", "mn", "k", 200, 300, 96, 1, "f32"),
    ("e2m3", "k", "k", 300, 520, 256, 2, "bf16"),
    ("e2m3", "k", "k", 200, 384, 384, 1, "f32"),
    ("e3m2", "k", "k", 513, 700, 512, 2, "bf16"),
    ("e3m2", "k", "k", 100, 300, 128, 1, "f32"),   # sums reach past the f16 range
    ("e2m1", "k", "k", 300, 520, 256, 2, "bf16"),
    ("e2m1", "k", "k", 1000, 1100, 640, 0, "bf16"),
    ("e2m1", "k", "k", 64, 256, 128, 1, "f32"),
    ("e2m1", "k", "k", 200, 300, 96, 1, "f32"),      # K not a multiple of the 256-K stage
    ("nvf4", "k", "k", 300, 520, 256, 2, "bf16"),
    ("nvf4", "k", "k", 513, 1100, 320, 0, "bf16"),   # 20 scales per row: a padded last stage
    ("nvf4", "k", "k", 100, 300, 64, 1, "f32"),
    ("nvf4", "k", "k", 256, 1024, 1024, 2, "bf16"),
]


@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out", MX_FORMATS)
def test_block_scaled_formats_full_compare(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out):
    x = make_case(dtype, am, bm, M, N, K, dist="codes" if dtype in syn.PACKED_BITS else "normal1", seed=M + K)
    _check_full(tcg, oracle_mod, x, out, "f32", cg)


@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out", [c for c in MX_FORMATS if c[0] in ("e2m1", "nvf4")])
def test_packed_fp4_copy_thread_staging(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out):
    # the packed-FP4 kinds' scales staged by a dedicated copy thread
    # (tcgen05.cp + commit to the slot's barrier) instead of the MMA thread
    x = make_case(dtype, am, bm, M, N, K, dist="codes", seed=M + K + 1)
    _check_full(tcg, oracle_mod, x, out, "f32", cg, sf_staging=3)
    with pytest.raises(tcg.TcgError):   # no tcgen05.st scale warps for these kinds
        run_gpu(tcg, x, out=out, cta_group=cg, sf_staging=1)


@pytest.mark.parametrize("dtype,one", [("e2m1", 0x2), ("e2m3", 0x08), ("e3m2", 0x0C), ("nvf4", 0x2)])
def test_packed_identity_reads_every_code_in_place(tcg, oracle_mod, dtype, one):
    """A = I (the code of 1.0 on the diagonal, scales 2^0) and B random codes:
    D[m, n] = B[n, m] decoded, exactly.  Pins how TMA expands the packed rows
    into shared memory and where the MMA reads each code, bit for bit."""
    bits = syn.PACKED_BITS[dtype]
    n, N = 256, 384
    A = syn.pack(np.where(np.eye(n, dtype=bool), one, 0).astype(np.uint8), bits)
    codes = syn.codes((N, n), 41 + bits, bits)
    B = syn.pack(codes, bits)
    nv = dtype == "nvf4"  # scales of one: e8m0 127 per 32, or unsigned E4M3 0x38 per 16
    SFA = np.full((n, n // (16 if nv else 32)), 0x38 if nv else 127, np.uint8)
    SFB = np.full((N, n // (16 if nv else 32)), 0x38 if nv else 127, np.uint8)
    D = torch.full((n, N), float("nan"), dtype=torch.float32, device="cuda")
    t = {"e2m1": tcg.IN_E2M1, "e2m3": tcg.IN_E2M3, "e3m2": tcg.IN_E3M2, "nvf4": tcg.IN_NVF4}[dtype]
    tcg.gemm(n, N, n, t, to_device(A), 0, n, to_device(B), 0, n, D, 0, N, 0, SFA=to_device(SFA), SFB=to_device(SFB))
    assert tcg.check() == 0
    expect = oracle_mod.decode(codes, oracle_mod.E2M1 if dtype in ("e2m1", "nvf4") else
                               oracle_mod.E2M3 if dtype == "e2m3" else oracle_mod.E3M2).T
    assert np.array_equal(D.double().cpu().numpy(), expect)


def test_named_fp6_fp4_entry_points(tcg, oracle_mod):
    for fmt, dtype in ((tcg.IN_E3M2, "e3m2"), (tcg.IN_E2M3, "e2m3"), (None, "e2m1"), ("nv", "nvf4")):
        x = make_case(dtype, "k", "k", 256, 320, 256, dist="codes", seed=5)
        D = torch.full((256, 320), float("nan"), dtype=torch.bfloat16, device="cuda")
        args = (256, 320, 256, to_device(x["A"]), 0, 256, to_device(x["B"]), 0, 256, to_device(x["SFA"]),
                to_device(x["SFB"]), D, 2, 320, 0)
        if fmt is None:
            tcg.gemm_mxf4_blockscaled(*args)
        elif fmt == "nv":
            tcg.gemm_nvf4_blockscaled(*args)
        else:
            tcg.gemm_mxf6_blockscaled(fmt, *args)
        assert tcg.check() == 0
        ref, S = oracle_rows(oracle_mod, x)
        assert_parity(D.double().cpu().numpy(), ref, S, TAU["f32"], dtype, "bf16")


def test_identity_gives_b_exactly(tcg, oracle_mod):
    # A = I: every D row is a B row, exact in bf16 out; pins the output layout.
    n, N = 256, 384
    A = syn.to_bits(np.eye(n), "bf16")
    b = syn.draw((n, N), 3, "uniform", n)
    B = syn.lay_out_b(syn.to_bits(b, "bf16"), "mn")
    D = torch.zeros((n, N), dtype=torch.bfloat16, device="cuda")
    tcg.gemm(n, N, n, 1, to_device(A), 0, n, to_device(B), 1, N, D, 2, N, 0, cta_group=2)
    assert tcg.check() == 0
    bdec = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(D.double().cpu().numpy(), bdec)


def test_permutation_rows_land_in_place(tcg):
    n, N = 512, 256
    perm = np.random.default_rng(9).permutation(n)
    P = syn.to_bits(np.eye(n)[perm], "f16")
    b = syn.draw((n, N), 4, "uniform", n)
    B = syn.lay_out_b(syn.to_bits(b, "f16"), "k")
    D = torch.zeros((n, N), dtype=torch.float32, device="cuda")
    tcg.gemm(n, N, n, 0, to_device(P), 0, n, to_device(B), 0, n, D, 0, N, 0, cta_group=1)
    assert tcg.check() == 0
    bdec = torch.from_numpy(B.view(np.int16)).view(torch.float16).double().numpy().T
    assert np.array_equal(D.double().cpu().numpy(), bdec[perm])


def test_blockscaled_identity_pins_scale_placement(tcg):
    # A = I in e4m3 with per-(row, 32-block) scales: D[m,n] =
    # 2^(sfa[m, m//32] + sfb[n, m//32] - 254) * B[m,n]; any misplaced scale
    # byte (lane, column, replica or SF id) changes an output by a power of two.
    n, N = 256, 448
    A = syn.to_bits(np.eye(n), "e4m3")
    b = syn.draw((n, N), 21, "normal1", n)
    B = syn.lay_out_b(syn.to_bits(b, "e4m3"), "k")
    rng = np.random.default_rng(22)
    SFA = (127 + rng.integers(-5, 6, size=(n, n // 32))).astype(np.uint8)
    SFB = (127 + rng.integers(-5, 6, size=(N, n // 32))).astype(np.uint8)
    bdec = torch.from_numpy(B).view(torch.float8_e4m3fn).double().numpy().T
    m = np.arange(n)
    expo = SFA[m, m // 32].astype(np.int64)[:, None] + SFB[:, m // 32].T.astype(np.int64) - 254
    ref = np.ldexp(bdec, expo)
    for cg in (1, 2):
        for staging in (1, 2, 3):  # tcgen05.st by scale warps / tcgen05.cp by the MMA thread / by a cp thread
            D = torch.zeros((n, N), dtype=torch.float32, device="cuda")
            tcg.gemm(n, N, n, 3, to_device(A), 0, n, to_device(B), 0, n, D, 0, N, 0, SFA=to_device(SFA),
                     SFB=to_device(SFB), cta_group=cg, sf_staging=staging)
            assert tcg.check() == 0
            assert np.array_equal(D.double().cpu().numpy(), ref), f"cta_group {cg} staging {staging}"


@pytest.mark.parametrize("staging", [1, 2, 3])
@pytest.mark.parametrize("am,bm,M,N,K,cg", [("k", "k", 300, 520, 256, 2), ("k", "k", 520, 300, 208, 1),
                                            ("mn", "mn", 200, 300, 256, 1), ("mn", "k", 260, 460, 640, 2),
                                            ("k", "k", 1100, 1300, 1024, 2), ("k", "mn", 520, 600, 384, 2),
                                            ("mn", "mn", 300, 300, 256, 2)])
def test_blockscaled_scale_staging_modes(tcg, oracle_mod, am, bm, M, N, K, cg, staging):
    # every explicit scale path: tcgen05.st by the scale warps (1), and
    # tcgen05.cp .32x128b.warpx4 issued by the MMA thread (2) or by a
    # dedicated thread that commits to a per-slot barrier (3); the larger
    # case runs many k-blocks per tile through every scale slot
    x = make_case("e4m3", am, bm, M, N, K, seed=M + 3 * N + K)
    _check_full(tcg, oracle_mod, x, "f32", "f32", cg, sf_staging=staging)


@pytest.mark.parametrize("staging", [2, 3])
@pytest.mark.parametrize("out", ["bf16", "f16"])
def test_blockscaled_pair_early_release(tcg, oracle_mod, staging, out):
    # one TMEM accumulator per CTA pair: the eight epilogue warps read it into
    # registers and release it before storing; 90 pair tiles on at most 76
    # clusters, so some clusters reuse the accumulator for a second tile
    x = make_case("e4m3", "k", "k", 2304, 2560, 256, seed=61 + staging)
    _check_full(tcg, oracle_mod, x, out, "f32", 2, sf_staging=staging)


# Split-K / stream-K: dtype, a_major, b_major, M, N, K, cta_group, out,
# split_k (-1 = stream-K, 0 = the library's choice, n >= 2 = fixed split).
# Explicit splits that do not divide the K blocks give uneven K ranges; the
# auto cases are long-K few-tile problems for which the library picks stream-K.
SPLIT = [
    ("bf16", "k", "k", 16, 1000, 2048, 1, "bf16", -1),
    ("bf16", "k", "k", 16, 1000, 8192, 1, "bf16", 0),
    ("bf16", "k", "mn", 1, 520, 1024, 1, "f32", 3),
    ("bf16", "k", "mn", 5, 2000, 4096, 0, "f32", 0),
    ("f16", "k", "k", 24, 600, 1536, 1, "f16", 3),
    ("bf16", "k", "k", 1000, 16, 4096, 1, "bf16", -1),
    ("bf16", "k", "k", 100, 300, 1000, 1, "bf16", 7),
    ("bf16", "mn", "k", 200, 700, 1536, 2, "bf16", -1),
    ("bf16", "k", "k", 256, 512, 4096, 2, "f16", -1),
    ("f16", "k", "k", 128, 256, 2048, 1, "f16", 5),
    ("tf32", "k", "k", 64, 300, 1024, 1, "f32", 4),
    ("tf32", "mn", "k", 36, 130, 520, 1, "bf16", -1),
    ("e4m3", "k", "k", 16, 520, 2048, 1, "bf16", -1),
    ("e4m3", "k", "k", 16, 520, 16384, 1, "bf16", 0),
    ("e4m3", "k", "k", 300, 512, 1024, 2, "bf16", 3),
    ("e4m3", "k", "mn", 64, 608, 4096, 2, "f32", -1),
]


@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out,split", SPLIT)
def test_split_k(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out, split):
    x = make_case(dtype, am, bm, M, N, K, seed=7 * M + N + K)
    # twice: the second call reuses the first one's workspace
    for _ in range(2):
        _check_full(tcg, oracle_mod, x, out, "f32", cg, split_k=split)


def test_split_k_workspace_survives_shape_changes(tcg, oracle_mod):
    # one stream, different shapes and splits back to back, then the first again
    cases = [make_case("bf16", "k", "k", 16, 1000, 2048, seed=91), make_case("bf16", "k", "k", 120, 384, 3072, seed=92)]
    for x, split in [(cases[0], 4), (cases[1], 6), (cases[0], -1), (cases[1], 2)]:
        _check_full(tcg, oracle_mod, x, "bf16", "f32", 1, split_k=split)
        assert tcg.last_launch_count() == 2  # the GEMM and the partial-tile reduction
    _check_full(tcg, oracle_mod, cases[1], "bf16", "f32", 1, split_k=1)
    assert tcg.last_launch_count() == 1


# Few rows of A against more columns than 64 x SMs: the library swaps the
# operands (D^T = B^T A^T on 128 x 32 tiles) and stores D transposed.
# dtype, b_major, M, K, out, split_k, extra columns of D's leading dimension
TRANSPOSED = [
    ("bf16", "k", 20, 1000, "bf16", 0, 0),
    ("bf16", "k", 1, 200, "f32", 0, 0),
    ("bf16", "mn", 16, 392, "f16", 0, 0),
    ("f16", "k", 32, 136, "f32", 0, 0),
    ("bf16", "k", 16, 520, "bf16", 0, 3),     # odd leading dimension of D
    ("bf16", "k", 7, 2048, "f32", -1, 1),     # stream-K: partial tiles reduced into the transposed D
    ("f16", "mn", 24, 1536, "bf16", 3, 0),    # fixed split
]


@pytest.mark.parametrize("dtype,bm,M,K,out,split,pad", TRANSPOSED)
def test_transposed_few_row_path(tcg, oracle_mod, dtype, bm, M, K, out, split, pad):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 64 * sms + 77  # ragged in the 128-row swapped tiles
    x = make_case(dtype, "k", bm, M, N, K, seed=M + K)
    _check_full(tcg, oracle_mod, x, out, "f32", 0, ldd=N + pad, split_k=split)
    plan = tcg.last_plan_string()
    assert "operands swapped" in plan and "tile 128x32" in plan, plan
    if split == -1:
        assert "stream-K" in plan, plan


def test_plan_choices_for_few_row_and_narrow_problems(tcg, oracle_mod):
    # skinny 64-column tiles in one pass; narrow 32-column tiles under stream-K
    x = make_case("bf16", "k", "k", 16, 4096, 1024, seed=61)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    assert "tile 128x64" in tcg.last_plan_string() and "swapped" not in tcg.last_plan_string()
    # 100 rows: 64-column tiles while they fit in one wave, else 128 x 256
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    x = make_case("bf16", "k", "k", 100, 2000, 512, seed=63)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    assert "tile 128x64" in tcg.last_plan_string(), tcg.last_plan_string()
    x = make_case("bf16", "k", "k", 100, 64 * sms + 100, 64, seed=64)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    assert "tile 128x256" in tcg.last_plan_string(), tcg.last_plan_string()
    # CTA pairs: 256 x 128 pair tiles while the 256 x 256 ones would fill at
    # most a quarter of the SMs, else 256 x 256
    x = make_case("bf16", "k", "mn", 300, 1100, 512, seed=65)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    assert "cta_group 2, tile 256x128" in tcg.last_plan_string(), tcg.last_plan_string()
    x = make_case("f16", "k", "k", 2100, 1100, 64, seed=66)   # 9 x 5 = 45 pair tiles > sms / 4
    _check_full(tcg, oracle_mod, x, "f16", "f32", 0)
    assert "cta_group 2, tile 256x256" in tcg.last_plan_string(), tcg.last_plan_string()
    x = make_case("bf16", "k", "k", 4096, 16, 8192, seed=62)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    plan = tcg.last_plan_string()
    assert "tile 128x32" in plan and "stream-K" in plan and "swapped" not in plan, plan


# rows, K, tile rows, byte offset of the plain scales, byte offset of the image.
# K = 200 / 1000 (kblocks 7 / 32): byte loads / word loads (the row stride is
# not a multiple of 16 bytes); K = 1024, 8192: 16-byte loads; offset scales:
# byte loads; offset image: word stores; K = 1664: a partial group of K steps.
PREPARE_CASES = [(300, 200, 128, 0, 0), (8192, 8192, 224, 0, 0), (500, 1024, 256, 0, 0),
                 (260, 1000, 224, 0, 0), (129, 1024, 128, 1, 0), (200, 1024, 224, 0, 4),
                 (384, 1664, 128, 0, 0), (1, 32, 224, 0, 0)]


def _plain_and_image(tcg, rows, K, tile, off, ioff, seed):
    kb = -(-K // 32)
    sf = np.random.default_rng(seed).integers(0, 255, size=(rows, kb)).astype(np.uint8)
    sf_dev = torch.zeros(rows * kb + 16, dtype=torch.uint8, device="cuda")
    sf_dev[off:off + rows * kb] = to_device(sf.reshape(-1))
    nbytes = tcg.mxf8_scale_image_bytes(rows, K, tile)
    img = torch.full((nbytes + 16,), 0xAB, dtype=torch.uint8, device="cuda")
    return sf, sf_dev[off:], img, img[ioff:ioff + nbytes]


@pytest.mark.parametrize("rows,K,tile,off,ioff", PREPARE_CASES)
def test_scale_prepare_kernel_matches_oracle_image(tcg, rows, K, tile, off, ioff):
    from oracle import layouts as L
    sf, sf_dev, img_all, img = _plain_and_image(tcg, rows, K, tile, off, ioff, rows + K)
    tcg.mxf8_prepare_scales(sf_dev, rows, K, tile, img)
    assert tcg.check() == 0
    exp = L.sf_prepare(sf, rows, -(-K // 32), tile).reshape(-1)
    assert np.array_equal(img.cpu().numpy(), exp), (rows, K, tile)
    rest = torch.cat([img_all[:ioff], img_all[ioff + exp.size:]]).cpu().numpy()
    assert (rest == 0xAB).all(), "wrote outside the image"


@pytest.mark.parametrize("M,N,K,tn", [(8192, 8192, 8192, 224), (300, 520, 200, 256), (0, 300, 256, 224)])
def test_scale_prepare_ab_matches_two_calls(tcg, M, N, K, tn):
    from oracle import layouts as L
    kb = -(-K // 32)
    sfa, sfa_dev, _, ia = _plain_and_image(tcg, M, K, 128, 0, 0, 7 + M)
    sfb, sfb_dev, _, ib = _plain_and_image(tcg, N, K, tn, 0, 0, 8 + N)
    tcg.mxf8_prepare_scales_ab(sfa_dev if M else None, M, ia if M else None, sfb_dev, N, tn, ib, K)
    assert tcg.check() == 0
    assert tcg.last_launch_count() == 1
    if M:
        assert np.array_equal(ia.cpu().numpy(), L.sf_prepare(sfa, M, kb, 128).reshape(-1))
    assert np.array_equal(ib.cpu().numpy(), L.sf_prepare(sfb, N, kb, tn).reshape(-1))


def test_prepared_scale_images_path(tcg, oracle_mod):
    x = make_case("e4m3", "k", "k", 384, 600, 320, seed=5)
    M, N, K = 384, 600, 320
    tn = tcg.mxf8_tile_n(M, N, K, 0, 2)
    ia = torch.zeros(tcg.mxf8_scale_image_bytes(M, K, 128), dtype=torch.uint8, device="cuda")
    ib = torch.zeros(tcg.mxf8_scale_image_bytes(N, K, tn), dtype=torch.uint8, device="cuda")
    tcg.mxf8_prepare_scales(to_device(x["SFA"]), M, K, 128, ia)
    tcg.mxf8_prepare_scales(to_device(x["SFB"]), N, K, tn, ib)
    D = run_gpu(tcg, x, out="f32", cta_group=2, sf_img=(ia, ib))
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(D[:M, :N].double().cpu().numpy(), ref, S, TAU["f32"], "prepared images")


def test_padded_leading_dims_and_unaligned_output(tcg, oracle_mod):
    x = make_case("bf16", "k", "k", 200, 300, 128, seed=3, extra_pad=2)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 1, ldd=307)   # odd ldd: scalar stores
    x = make_case("f16", "mn", "k", 200, 300, 128, seed=4, extra_pad=1)
    _check_full(tcg, oracle_mod, x, "f32", "f32", 2, ldd=320)


def test_absurd_tile_counts_are_refused_before_any_launch(tcg):
    # (2^30 - 1)^2 outputs: 2^44 pair tiles, far beyond 32-bit tile indices;
    # refused on the host (the pointers are never touched)
    M = N = (1 << 30) - 1
    rc = tcg.gemm(M, N, 64, 1, 0x10000, 0, 64, 0x20000, 0, 64, 0x30000, 2, N, 0, check=False)
    assert rc == tcg.ERR_UNSUPPORTED
    assert "tiles" in tcg.last_error_string()
    assert tcg.check() == 0


def test_phase_trace(tcg, oracle_mod):
    # 1024 x 1024 x 512 on 256 x 128 pair tiles: 32 clusters, one tile each
    import re
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros((sms, 10), dtype=torch.int64, device="cuda")
    x = make_case("bf16", "k", "k", 1024, 1024, 512, seed=72)
    tcg.trace_next(buf, sms)
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    plan = tcg.last_plan_string()
    m = re.search(r"cta_group (\d), tile (\d+)x(\d+), (\d+) clusters", plan)
    cg, clusters = int(m.group(1)), int(m.group(4))
    tiles = -(-1024 // int(m.group(2))) * -(-1024 // int(m.group(3)))
    t = buf.cpu().numpy()
    ctas = cg * clusters
    assert np.all(t[ctas:] == 0)                        # no stamps beyond the grid
    units = 0
    for c in range(ctas):
        e, su, pr, fu, lc, ep, ex, un, c0, c1 = t[c]
        assert 0 < e <= su <= pr and su <= ep <= ex and ex - e < 10**9, (c, t[c])
        # cycles over nanoseconds: an SM clock between 0.5 and 2.5 GHz
        assert 0.5 * (ex - e) <= c1 - c0 <= 2.5 * (ex - e), (c, t[c])
        if c % cg == 0:                                 # the MMA warp of the leader
            assert pr <= fu <= lc <= ep and un >= 1, (c, t[c])
            units += un
    assert units == tiles
    # the request covers one launch only
    buf.zero_()
    _check_full(tcg, oracle_mod, x, "bf16", "f32", 0)
    assert int(buf.abs().sum().item()) == 0


def test_k_zero_zeroes_d_and_empty_is_noop(tcg):
    D = torch.full((64, 80), 7.0, dtype=torch.float32, device="cuda")
    tcg.gemm_bf16(64, 80, 0, 0, 0, 0, 0, 0, 0, D, 0, 80, 0)
    assert tcg.check() == 0
    assert torch.count_nonzero(D).item() == 0
    D.fill_(7.0)
    tcg.gemm_bf16(0, 80, 64, 0, 0, 0, 0, 0, 0, D, 0, 80, 0)
    tcg.gemm_bf16(64, 0, 64, 0, 0, 0, 0, 0, 0, D, 0, 80, 0)
    assert tcg.check() == 0
    assert torch.all(D == 7.0)


def test_named_entry_points(tcg, oracle_mod):
    x = make_case("bf16", "k", "mn", 256, 384, 192, seed=8)
    D = torch.zeros((256, 384), dtype=torch.bfloat16, device="cuda")
    tcg.gemm_bf16(256, 384, 192, to_device(x["A"]), 0, x["lda"], to_device(x["B"]), 1, x["ldb"], D, 2, 384, 0)
    assert tcg.check() == 0
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(D.double().cpu().numpy(), ref, S, TAU["f32"], "gemm_bf16", "bf16")
    x = make_case("e4m3", "k", "k", 256, 384, 256, seed=9)
    D = torch.zeros((256, 384), dtype=torch.bfloat16, device="cuda")
    tcg.gemm_mxf8_blockscaled(256, 384, 256, to_device(x["A"]), 0, x["lda"], to_device(x["B"]), 0, x["ldb"],
                              to_device(x["SFA"]), to_device(x["SFB"]), D, 2, 384, 0)
    assert tcg.check() == 0
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(D.double().cpu().numpy(), ref, S, TAU["f32"], "gemm_mxf8_blockscaled", "bf16")


# ------------------------------------------------------------- 256 x 384 pair tiles

# Packed-FP4 CTA pairs over at least 300 tiles of 256 x 384 take the two-MMA
# tile (N = 256 then N = 128 per K step).  M = 2600 leaves the last pair
# tile's second CTA wholly beyond M; N = 10668 ends on a tile whose 300
# columns reach into the second MMA's first CTA half.
WIDE = [
    # dtype, K, out, split
    ("e2m1", 320, "bf16", 0),
    ("e2m1", 256, "f32", 0),
    ("e2m1", 1024, "f32", 3),
    ("nvf4", 512, "bf16", 0),
    ("nvf4", 256, "f32", 0),
    ("nvf4", 768, "bf16", 2),
]


@pytest.mark.parametrize("staging", [0, 3])
@pytest.mark.parametrize("dtype,K,out,split", WIDE)
def test_wide_pair_tiles_sampled_rows(tcg, oracle_mod, dtype, K, out, split, staging):
    M, N = 2600, 27 * 384 + 300
    x = make_case(dtype, "k", "k", M, N, K, dist="codes", seed=K + len(dtype))
    assert tcg.tile_n(IN_TYPE[dtype], M, N, K, 0, 0) == 384
    D = run_gpu(tcg, x, out=out, cta_group=0, split_k=split, sf_staging=staging)
    plan = tcg.last_plan_string()
    assert "cta_group 2, tile 256x384" in plan, plan
    rows = sample_rows(M, n=16, seed=K)
    got = D[rows, :N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    assert_parity(got, ref, S, TAU["f32"], f"{dtype} 256x384 split {split}", out)


def test_eight_bit_and_fp6_keep_256_wide_pair_tiles(tcg, oracle_mod):
    M, N, K = 2600, 27 * 384 + 300, 256
    for dtype in ("e4m3", "e2m3"):
        assert tcg.tile_n(IN_TYPE[dtype], M, N, K, 0, 0) == 256
    x = make_case("e4m3", "k", "k", M, N, K, seed=5)
    D = run_gpu(tcg, x, out="bf16", cta_group=0)
    assert "cta_group 2, tile 256x256" in tcg.last_plan_string(), tcg.last_plan_string()
    rows = sample_rows(M, n=6, seed=5)
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    assert_parity(D[rows, :N].double().cpu().numpy(), ref, S, TAU["f32"], "e4m3 256x256", "bf16")


# ------------------------------------------------------------- fragment epilogue

# epilogue = 2: 16-bit outputs drained with tcgen05.ld .16x256b and written to
# the staging tile with stmatrix.  Every variant that stages 16-bit outputs:
# 128 x 256 and pair tiles (two accumulators), 256 x 128 pair tiles, the
# 64-column skinny and 32-column narrow tiles, TF32, MXFP8 pairs (one
# accumulator read whole before release, eight warps) and the 256 x 384 FP4
# pair tile; ragged M and N throughout.
FRAG = [
    # dtype, am, bm, M, N, K, cg, out  (N a multiple of 8: 16-byte output rows)
    ("bf16", "k", "k", 300, 520, 200, 1, "bf16"),
    ("f16", "mn", "k", 513, 1096, 136, 2, "f16"),
    ("bf16", "k", "mn", 300, 1096, 512, 0, "bf16"),
    ("bf16", "k", "k", 100, 520, 640, 1, "f16"),
    ("bf16", "k", "k", 700, 24, 1000, 1, "bf16"),
    ("tf32", "k", "k", 300, 520, 200, 2, "bf16"),
    ("e4m3", "k", "k", 300, 1096, 256, 2, "bf16"),
    ("e4m3", "mn", "k", 260, 232, 160, 1, "f16"),
    ("e2m1", "k", "k", 2600, 27 * 384 + 296, 256, 0, "bf16"),
]


@pytest.mark.parametrize("dtype,am,bm,M,N,K,cg,out", FRAG)
def test_fragment_epilogue_matches_row_epilogue_bit_for_bit(tcg, oracle_mod, dtype, am, bm, M, N, K, cg, out):
    x = make_case(dtype, am, bm, M, N, K, dist="codes" if dtype in syn.PACKED_BITS else "uniform", seed=M + N)
    rows_d = run_gpu(tcg, x, out=out, cta_group=cg, epilogue=1)
    assert "stmatrix" not in tcg.last_plan_string()
    frag_d = run_gpu(tcg, x, out=out, cta_group=cg, epilogue=2)
    assert "16x256b + stmatrix epilogue" in tcg.last_plan_string(), tcg.last_plan_string()
    assert torch.equal(rows_d.view(torch.int16), frag_d.view(torch.int16))
    rows = sample_rows(M, n=8, seed=N) if M > 512 else list(range(M))
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    assert_parity(frag_d[rows, :N].double().cpu().numpy(), ref, S, TAU["f32"], f"{dtype} fragment epilogue", out)


def test_fragment_epilogue_request_is_ignored_where_it_does_not_apply(tcg, oracle_mod):
    # fp32 output, and a 16-bit output whose ldd is not a 16-byte multiple
    # (per-lane row stores, no staging tile): the row path serves both
    x = make_case("bf16", "k", "k", 300, 520, 200, seed=3)
    run_gpu(tcg, x, out="f32", cta_group=1, epilogue=2)
    assert "stmatrix" not in tcg.last_plan_string()
    D = torch.full((300, 523), float("nan"), dtype=torch.bfloat16, device="cuda")
    run_gpu(tcg, x, out="bf16", cta_group=1, epilogue=2, ldd=523, D=D)
    assert "stmatrix" not in tcg.last_plan_string()
    ref, S = oracle_rows(oracle_mod, x)
    assert_parity(D[:, :520].double().cpu().numpy(), ref, S, TAU["f32"], "row path", "bf16")


# ------------------------------------------------------------- full-size workloads

FULL = ["tile_f16_128x128x64", "bf16_4096_kmn_cta1", "tf32_2048x2048x8192", "bf16_8192_cta2",
        "f16acc_8192_cta2", "mxf8_8192", "bf16_skinny_m16", "bf16_skinny_m128", "mxf6_e2m3_8192", "mxf4_8192",
        "nvf4_8192"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workloads_sampled_rows(tcg, oracle_mod, name):
    w = syn.WORKLOADS[name]
    x = syn.make_inputs(w)
    x["w"] = w
    D = run_gpu(tcg, x, out=w.out, acc=w.acc, cta_group=w.cta_group)
    rows = sample_rows(w.M) if w.M > 256 else list(range(w.M))
    got = D[rows, :w.N].double().cpu().numpy()
    ref, S = oracle_rows(oracle_mod, x, rows=rows)
    ratio = assert_parity(got, ref, S, TAU[w.acc], name, w.out)
    print(f"{name}: max err/S {ratio:.3e} over {len(rows)} rows")


def test_one_pass_plans_agree_bit_for_bit(tcg):
    # every one-pass plan accumulates each output over K in the same order of
    # K-16 MMA steps, whatever its tile: CTA pairs, single CTAs, the skinny
    # 64-column tiles (few rows) and the narrow 32-column tiles (few columns)
    # give identical fp32 outputs on the rows / columns they share
    g = torch.Generator().manual_seed(77)
    M, N, K = 1000, 1100, 640
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()

    def run(m, n, cg):
        D = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        tcg.gemm(m, n, K, tcg.IN_BF16, A, 0, K, B, 0, K, D, tcg.F32, n, tcg.F32, cta_group=cg, split_k=1)
        assert tcg.check() == 0
        return D, tcg.last_plan_string()

    ref, p2 = run(M, N, 2)
    assert "cta_group 2" in p2, p2
    for m, n, cg, tile in ((M, N, 1, "128x256"), (100, N, 0, "128x64"), (20, N, 0, "128x64"), (M, 24, 0, "128x32")):
        D, plan = run(m, n, cg)
        assert tile in plan, plan
        assert torch.equal(D, ref[:m, :n]), plan


def _rows_of(x, m):
    # the first m rows of a case (A and its scales), same B
    y = dict(x)
    y["M"] = m
    y["A"] = x["A"][:m]
    if "SFA" in x:
        y["SFA"] = x["SFA"][:m]
    return y


@pytest.mark.parametrize("dtype,M,N,K", [("e4m3", 1000, 1100, 256), ("e2m1", 2600, 27 * 384 + 300, 256),
                                         ("nvf4", 2600, 27 * 384 + 300, 512)])
def test_block_scaled_plans_agree_bit_for_bit(tcg, dtype, M, N, K):
    # the same operands through different tiles: MXFP8 CTA pairs and single
    # CTAs; packed FP4 on 256 x 384 pair tiles (two MMAs per K step, chosen
    # for many tiles) and, for the first 256 rows alone, 256 x 256 pair tiles
    x = make_case(dtype, "k", "k", M, N, K, dist="codes" if dtype in syn.PACKED_BITS else "normal1", seed=M + K)
    ref = run_gpu(tcg, x, out="f32", cta_group=0, split_k=1)
    plan_ref = tcg.last_plan_string()
    if dtype == "e4m3":
        D = run_gpu(tcg, x, out="f32", cta_group=1, split_k=1)
        assert "cta_group 1" in tcg.last_plan_string() and "cta_group 2" in plan_ref
        assert torch.equal(D, ref)
    else:
        assert "tile 256x384" in plan_ref, plan_ref
        D = run_gpu(tcg, _rows_of(x, 256), out="f32", cta_group=0, split_k=1)
        assert "tile 256x256" in tcg.last_plan_string(), tcg.last_plan_string()
        assert torch.equal(D, ref[:256]), tcg.last_plan_string()
