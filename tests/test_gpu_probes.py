"""GPU layout probes, bit-exact against the pages' layout rules as restated
in ``oracle.layouts`` (and the pages' worked examples in
``tests/golden/page_examples.json``)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import layouts as L

pytestmark = pytest.mark.gpu
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


@pytest.fixture(scope="module")
def tcg():
    assert torch.cuda.is_available(), "GPU tests need a GPU"
    from blackwell_tensor_core_swizzled_gb300 import build
    build.build()
    import blackwell_tensor_core_swizzled_gb300 as m
    return m


def _u32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


def _np(t):
    return t.cpu().numpy().view(np.uint32)


# ------------------------------------------------------------- TMEM round trips

def test_tmem_roundtrip_layout_b_page_example(tcg):
    ex = GOLDEN["tmem_st_ld_layout_b"]
    x = np.arange(8192, dtype=np.float32).reshape(ex["shape"])
    inp = _u32(x.view(np.uint32))
    out = torch.zeros_like(inp)
    tcg.probe_tmem_roundtrip(inp, out, 64)
    assert tcg.check() == 0
    assert np.array_equal(_np(out).view(np.float32).reshape(128, 64), x)


@pytest.mark.parametrize("ncols", [1, 2, 4, 8, 16, 32, 64])
def test_tmem_roundtrip_random_bits(tcg, ncols):
    rng = np.random.default_rng(ncols)
    bits = rng.integers(0, 2**32, size=(128, ncols), dtype=np.uint64).astype(np.uint32)
    inp = _u32(bits)
    out = torch.zeros_like(inp)
    tcg.probe_tmem_roundtrip(inp, out, ncols)
    assert tcg.check() == 0
    assert np.array_equal(_np(out).reshape(128, ncols), bits)


def test_tmem_roundtrip_128x8_f16(tcg):
    # copy_async -> tcgen05_ldst page demonstration: a 128x8 fp16 tile through
    # 32x32b.x4 (two fp16 per 32-bit cell)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((128, 8)).astype(np.float16)
    inp = _u32(x.view(np.uint32).reshape(128, 4))
    out = torch.zeros_like(inp)
    tcg.probe_tmem_roundtrip(inp, out, 4)
    assert tcg.check() == 0
    assert np.array_equal(_np(out).reshape(128, 4).view(np.float16), x)


# ------------------------------------------------------------- tcgen05.cp

CP_ROWS = {0: 128, 1: 128, 2: 32, 3: 4}
CP_WORDS = {0: 8, 1: 4, 2: 4, 3: 8}


def _cp_expected(image, shape, origin, ldo, sdo, sw):
    # shape + 4: FP4 decompression, shape + 8: FP6; same source walk
    fmt = {0: None, 1: 4, 2: 6}[shape // 4]
    shape %= 4
    exp = np.full((128, 8), 0xDEADBEEF, dtype=np.uint32)
    r, w = np.meshgrid(np.arange(CP_ROWS[shape]), np.arange(CP_WORDS[shape]), indexing="ij")
    phys = L.cp_physical(origin, r, w, ldo, sdo, sw)
    vals = image[phys // 4]
    if fmt is not None:  # every 16-byte block of a row expands on its own
        vals = L.cp_decompress(vals.reshape(vals.shape[0], -1, 4), fmt).reshape(vals.shape)
    if shape in (0, 1):
        exp[:, :CP_WORDS[shape]] = vals
    elif shape == 2:  # 32x128b.warpx4: four replicas 32 lanes apart
        for q in range(4):
            exp[32 * q:32 * q + 32, :4] = vals
    else:  # 4x256b: lanes 0, 32, 64, 96
        for i in range(4):
            exp[32 * i, :] = vals[i]
    return exp


CP_CASES = [
    # shape, origin, ldo, sdo, swizzle, image_words
    (1, 0, 16, 128, 0, 512),       # the page's example (128x128b, (16, 128, 0))
    (0, 0, 256, 128, 0, 2048),     # unswizzled 8-word rows: words 4..7 at LDO
    (0, 0, 2048, 256, 0, 2048),
    (0, 0, 16, 256, 1, 2048),      # 32-byte rows, 256-byte period
    (0, 0, 16, 512, 2, 4096),      # 64-byte rows, 512-byte period
    (0, 0, 16, 1024, 3, 4096),     # 128-byte rows, 1024-byte period
    (0, 64, 16, 1024, 3, 4352),    # origin inside the first row: swizzle phase
    (1, 16, 16, 1024, 3, 4352),
    (0, 32, 16, 2048, 3, 8448),    # gaps between row groups
    (1, 48, 16, 512, 2, 4352),
    (2, 0, 16, 128, 0, 128),       # 32x128b.warpx4: the scale-factor staging shape
    (2, 0, 16, 1024, 3, 1024),
    (3, 0, 16, 128, 0, 64),        # 4x256b
]


@pytest.mark.parametrize("shape,origin,ldo,sdo,sw,words", CP_CASES)
def test_cp_walk_and_swizzle(tcg, shape, origin, ldo, sdo, sw, words):
    if shape == 1 and origin == 0 and sw == 0:
        image = np.arange(words, dtype=np.uint32)          # arange(512), as on the page
    else:
        image = (np.arange(words, dtype=np.uint32) * 2654435761) & 0xFFFFFFFF
        image = image.astype(np.uint32)
    img = _u32(image)
    out = torch.zeros((128, 8), dtype=torch.int32, device="cuda")
    tcg.probe_cp(img, words, shape, origin, ldo, sdo, sw, out)
    assert tcg.check() == 0
    got = _np(out)
    exp = _cp_expected(image, shape, origin, ldo, sdo, sw)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)[:6]
        raise AssertionError(f"mismatch at {bad.tolist()}: got {[hex(got[tuple(b)]) for b in bad]} "
                             f"exp {[hex(exp[tuple(b)]) for b in bad]}")
    if shape == 1 and origin == 0 and sw == 0:
        assert np.array_equal(got[:, :4], np.arange(512).reshape(128, 4))  # page: out == x


# FP4 / FP6 decompression ("tcgen05.cp" page, "Native FP4/FP6 decompression"):
# every shape with each format; random words, so the padding bytes are
# arbitrary and must not reach TMEM.
DECOMP_CASES = [
    (base + 4 * fmt, origin, ldo, sdo, sw, words)
    for fmt in (1, 2)
    for (base, origin, ldo, sdo, sw, words) in [
        (0, 0, 256, 128, 0, 2048), (1, 0, 16, 128, 0, 512), (2, 0, 16, 128, 0, 128), (3, 0, 16, 128, 0, 64),
        (0, 0, 16, 1024, 3, 4096), (1, 48, 16, 512, 2, 4352)]
]


@pytest.mark.parametrize("shape,origin,ldo,sdo,sw,words", DECOMP_CASES)
def test_cp_decompression(tcg, shape, origin, ldo, sdo, sw, words):
    image = np.random.default_rng(shape * 100 + sw).integers(0, 1 << 32, words, dtype=np.uint64).astype(np.uint32)
    out = torch.zeros((128, 8), dtype=torch.int32, device="cuda")
    tcg.probe_cp(_u32(image), words, shape, origin, ldo, sdo, sw, out)
    assert tcg.check() == 0
    got = _np(out)
    exp = _cp_expected(image, shape, origin, ldo, sdo, sw)
    if not np.array_equal(got, exp):
        bad = np.argwhere(got != exp)[:6]
        raise AssertionError(f"mismatch at {bad.tolist()}: got {[hex(got[tuple(b)]) for b in bad]} "
                             f"exp {[hex(exp[tuple(b)]) for b in bad]}")


# ------------------------------------------------------------- ld images

SHAPE_ID = {"32x32b": 0, "16x64b": 1, "16x128b": 2, "16x256b": 3}


@pytest.mark.parametrize("shape", list(SHAPE_ID))
@pytest.mark.parametrize("num", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("half", [0, 1])
def test_ld_register_images(tcg, shape, num, half):
    if shape == "32x32b" and half == 1:
        pytest.skip("32-row shape has no half")
    if L.ld_atom_extent(shape, num)[1] > 32:
        pytest.skip("wider than the 32-column image")
    image = (np.arange(128)[:, None] * 32 + np.arange(32)[None, :]).astype(np.uint32)
    out = torch.zeros((128, 4 * num), dtype=torch.int32, device="cuda")
    tcg.probe_ld_shape(_u32(image), SHAPE_ID[shape], num, half, out)
    assert tcg.check() == 0
    regs = L.ld_regs_per_lane(shape, num)
    got = _np(out).reshape(-1)[:128 * regs].reshape(128, regs)
    for warp in range(4):
        lane0 = 32 * warp + (16 * half if shape != "32x32b" else 0)
        exp = L.ld_image(shape, num, lambda row, col: image[lane0 + row, col])
        assert np.array_equal(got[32 * warp:32 * warp + 32], exp), (shape, num, half, warp)


# ------------------------------------------------------------- one MMA tile

def test_mma_tile_page_example_exact(tcg, oracle_mod):
    ex = GOLDEN["mma_four_k16"]
    rng = np.random.default_rng(ex["seed"])
    a = (rng.integers(-4, 5, (128, 64)) / 4).astype("float16")
    b = (rng.integers(-4, 5, (64, 64)) / 4).astype("float16")
    D = torch.zeros((128, 64), dtype=torch.float32, device="cuda")
    tcg.probe_mma_tile(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda(), 64, 64, 0, D)
    assert tcg.check() == 0
    got = D.cpu().numpy()
    np.testing.assert_allclose(got, a.astype("float32") @ b.astype("float32").T, rtol=ex["rtol"], atol=ex["atol"])
    ref, _ = oracle_mod.gemm(128, 64, 64, a.view(np.uint16), 1, 0, 64, b.view(np.uint16), 1, 0, 64)
    assert np.array_equal(got.astype(np.float64), ref)   # exact: quarter-integer sums


@pytest.mark.parametrize("N,K,bf16", [(128, 64, 0), (256, 64, 1), (16, 16, 0), (48, 32, 1)])
def test_mma_tile_random(tcg, oracle_mod, N, K, bf16):
    import synthetic as syn
    dt = "bf16" if bf16 else "f16"
    a = syn.to_bits(syn.draw((128, K), 100 + N, "uniform", K), dt)
    b = syn.to_bits(syn.draw((N, K), 200 + N, "uniform", K), dt)
    D = torch.zeros((128, N), dtype=torch.float32, device="cuda")
    tcg.probe_mma_tile(torch.from_numpy(a.view(np.int16)).cuda(), torch.from_numpy(b.view(np.int16)).cuda(),
                       N, K, bf16, D)
    assert tcg.check() == 0
    ref, S = oracle_mod.gemm(128, N, K, a, 2 if bf16 else 1, 0, K, b, 2 if bf16 else 1, 0, K)
    err = np.abs(D.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 2e-3 * S)


@pytest.mark.parametrize("N,K,bf16", [(64, 64, 0), (128, 32, 1), (256, 64, 0), (256, 16, 1)])
def test_mma_tile_weight_stationary(tcg, oracle_mod, N, K, bf16):
    # .ws with M = 128: Layout D (lane = row), so the same exact result as the
    # dense opcode; quarter-integer inputs make every sum exact in fp32
    rng = np.random.default_rng(N + K + bf16)
    a = (rng.integers(-4, 5, (128, K)) / 4).astype(np.float32)
    b = (rng.integers(-4, 5, (N, K)) / 4).astype(np.float32)
    dt = "bf16" if bf16 else "f16"
    import synthetic as syn
    ab, bb = syn.to_bits(a.astype(np.float64), dt), syn.to_bits(b.astype(np.float64), dt)
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    tcg.probe_mma_tile_ws(torch.from_numpy(ab.view(np.int16)).cuda(), torch.from_numpy(bb.view(np.int16)).cuda(),
                          N, K, bf16, D)
    assert tcg.check() == 0
    ref, _ = oracle_mod.gemm(128, N, K, ab, 2 if bf16 else 1, 0, K, bb, 2 if bf16 else 1, 0, K)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), ref)


# ------------------------------------------------------------- ldmatrix

def test_ldmatrix_x2_page_example(tcg):
    ex = GOLDEN["ldmatrix_x2_interleaved"]
    x = np.arange(128, dtype=np.uint32).reshape(16, 4, 2)
    out = torch.zeros((32, 12), dtype=torch.int32, device="cuda")
    tcg.probe_ldmatrix_x2(_u32(x.reshape(-1)), out)
    assert tcg.check() == 0
    expected = np.full((32, 12), ex["sentinel"], dtype=np.uint64)
    for lane in range(32):
        for k in range(2):
            for matrix in range(2):
                expected[lane, 8 * k + 2 * matrix] = x[2 * (lane // 4) + matrix, lane % 4, k]
    assert np.array_equal(_np(out).astype(np.uint64), expected)


@pytest.mark.parametrize("count", [1, 2, 4])
@pytest.mark.parametrize("trans", [False, True])
def test_stmatrix_rows_land_at_provider_addresses(tcg, count, trans):
    # rows scattered over a 1 KB buffer in a seeded order with gaps between them
    rng = np.random.default_rng(100 + 2 * count + int(trans))
    slots = rng.permutation(64)[:8 * count]
    row_off = (16 * slots).astype(np.uint32)
    regs = rng.integers(0, 2**32, size=(32, 4), dtype=np.uint64)
    out = torch.zeros(256, dtype=torch.int32, device="cuda")
    tcg.probe_stmatrix(_u32(regs.astype(np.uint32).reshape(-1)), _u32(row_off), count, trans, out)
    assert tcg.check() == 0
    rows = L.stmatrix_store([[int(v) for v in regs[l, :count]] for l in range(32)], count, trans)
    expected = np.zeros(256, dtype=np.uint64)
    for m in range(count):
        for r in range(8):
            expected[row_off[8 * m + r] // 4 + np.arange(4)] = rows[m][r]
    assert np.array_equal(_np(out).astype(np.uint64), expected)


@pytest.mark.parametrize("num", [1, 2, 4, 8])
@pytest.mark.parametrize("imm", [(16, 8), (16, 0), (0, 16), (16, 16)])
def test_split_16x32bx2_load_and_store(tcg, num, imm):
    il, ic = imm
    rng = np.random.default_rng(7 * num + il + ic)
    image = rng.integers(0, 2**32, size=(128, 32), dtype=np.uint64).astype(np.uint32)
    out_ld = torch.zeros(128 * num, dtype=torch.int32, device="cuda")
    out_st = torch.full((128 * 32,), -1, dtype=torch.int32, device="cuda")
    tcg.probe_ld_split(_u32(image.reshape(-1)), num, il, ic, out_ld, out_st)
    assert tcg.check() == 0
    got_ld = _np(out_ld).reshape(128, num)
    got_st = _np(out_st).reshape(128, 32)
    for w in range(4):
        exp = L.split_load(num, il, ic, lambda r, c: image[32 * w + r, c])
        assert np.array_equal(got_ld[32 * w:32 * w + 32], exp), (num, imm, w)
        t = 32 * w + np.arange(32)[:, None]
        regs = (0x10000 * t + np.arange(num)[None, :] + 1).astype(np.uint64)
        assert np.array_equal(got_st[32 * w:32 * w + 32].astype(np.uint64), L.split_store(regs, il, ic)), (num, imm, w)


# ------------------------------------------------------------- failure detection

def test_bounded_wait_reports_timeout_and_context_survives(tcg):
    assert tcg.check() == 0
    tcg.probe_wait_timeout(2_000_000)      # 2 ms on a barrier nobody arrives at
    assert tcg.check() == tcg.ERR_TIMEOUT
    assert tcg.check() == 0                # the error word was cleared
    vals = torch.arange(128 * 8, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(vals)
    tcg.probe_tmem_roundtrip(vals, out, 8)  # the context is still usable
    assert tcg.check() == 0 and torch.equal(out, vals)


# ------------------------------------------------------------- MMA from model-built images

from mma_image_cases import CASES as IMAGE_CASES, build_image, kstep as _kstep  # noqa: E402

_IN = {"f16": 0, "bf16": 1, "tf32": 2}
_ORACLE_T = {"f16": 1, "bf16": 2, "tf32": 0}


@pytest.mark.parametrize("case", IMAGE_CASES, ids=[c.name for c in IMAGE_CASES])
def test_mma_reads_oracle_layout_model(tcg, oracle_mod, case):
    """The oracle's operand walk (K-major and MN-major, swizzle modes 0..4)
    lays out A and B; the hardware's descriptor walk must read back exactly
    the logical operands: quarter-integer inputs make every sum exact, so the
    product must equal the oracle's float64 GEMM bit for bit."""
    import synthetic as syn
    ks = case.K // _kstep(case.dtype)
    rng = np.random.default_rng(len(case.name) * 7 + case.N)
    a = rng.integers(-4, 5, (128, case.K)) / 4.0
    b = rng.integers(-4, 5, (case.N, case.K)) / 4.0
    ab, bb = syn.to_bits(a, case.dtype), syn.to_bits(b, case.dtype)
    img_a = build_image(ab, case.a, case.dtype, ks)
    img_b = build_image(bb, case.b, case.dtype, ks)
    from mma_image_cases import issue_starts
    da, db = torch.from_numpy(img_a).cuda(), torch.from_numpy(img_b).cuda()
    opa = tcg.probe_operand(da, img_a.size, 0 if case.a.major == "k" else 1, case.a.ldo, case.a.sdo, case.a.swizzle,
                            issue_starts(case.a, 128, case.dtype, ks))
    opb = tcg.probe_operand(db, img_b.size, 0 if case.b.major == "k" else 1, case.b.ldo, case.b.sdo, case.b.swizzle,
                            issue_starts(case.b, case.N, case.dtype, ks))
    D = torch.full((128, case.N), float("nan"), dtype=torch.float32, device="cuda")
    tcg.probe_mma_image(opa, opb, _IN[case.dtype], case.N, ks, D)
    assert tcg.check() == 0
    t = _ORACLE_T[case.dtype]
    ref, _ = oracle_mod.gemm(128, case.N, case.K, ab, t, 0, case.K, bb, t, 0, case.K)
    got = D.cpu().numpy().astype(np.float64)
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)[:6]
        raise AssertionError(f"{case.name}: {int((got != ref).sum())} mismatches, first {bad.tolist()}: "
                             f"got {[got[tuple(i)] for i in bad]} ref {[ref[tuple(i)] for i in bad]}")


@pytest.mark.parametrize("N,K,bf16", [(128, 64, 0), (256, 64, 1), (64, 16, 0), (48, 32, 1)])
def test_mma_with_a_in_tmem(tcg, oracle_mod, N, K, bf16):
    """A written to tensor memory (Layout D: row m in lane m, two 16-bit values
    per column) and read by the MMA from there; quarter-integer inputs make
    every sum exact, so the product equals the oracle's bit for bit."""
    import synthetic as syn
    rng = np.random.default_rng(3 * N + K + bf16)
    a = rng.integers(-4, 5, (128, K)) / 4.0
    b = rng.integers(-4, 5, (N, K)) / 4.0
    dt = "bf16" if bf16 else "f16"
    ab, bb = syn.to_bits(a, dt), syn.to_bits(b, dt)
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    tcg.probe_mma_tmem_a(torch.from_numpy(ab.view(np.int16)).cuda(), torch.from_numpy(bb.view(np.int16)).cuda(),
                         N, K, bf16, D)
    assert tcg.check() == 0
    ref, _ = oracle_mod.gemm(128, N, K, ab, 2 if bf16 else 1, 0, K, bb, 2 if bf16 else 1, 0, K)
    assert np.array_equal(D.cpu().numpy().astype(np.float64), ref)


@pytest.mark.parametrize("N,K,bf16", [(64, 32, 0), (128, 64, 1), (256, 16, 0)])
@pytest.mark.parametrize("a_tmem", [0, 1])
def test_ws64_accumulator_and_tmem_a_banks(tcg, oracle_mod, N, K, bf16, a_tmem):
    """M = 64 weight-stationary tile: the raw 128-lane x N/2-column
    accumulator image equals the oracle product placed by the layout model
    (columns split into two banks at N/2).  With A in TMEM the two banks hold
    different A rows, so each bank's columns must come from its own bank."""
    import synthetic as syn
    rng = np.random.default_rng(7 * N + K + 2 * a_tmem + bf16)
    dt = "bf16" if bf16 else "f16"
    banks = rng.integers(-4, 5, (2, 64, K)) / 4.0
    if not a_tmem:
        banks[1] = banks[0]   # one A from shared memory serves both banks
    b = rng.integers(-4, 5, (N, K)) / 4.0
    ab = syn.to_bits(banks.reshape(128, K), dt)
    bb = syn.to_bits(b, dt)
    a_in = ab if a_tmem else ab[:64]
    out = torch.zeros((128, N // 2), dtype=torch.int32, device="cuda")
    tcg.probe_mma_ws64(torch.from_numpy(np.ascontiguousarray(a_in).view(np.int16)).cuda(), a_tmem,
                       torch.from_numpy(bb.view(np.int16)).cuda(), N, K, bf16, out)
    assert tcg.check() == 0
    got = out.cpu().numpy().view(np.float32).astype(np.float64)
    t = 2 if bf16 else 1
    expect = np.full((128, N // 2), np.nan)
    half = N // 2
    for bank in range(2):
        ref, _ = oracle_mod.gemm(64, N, K, ab[64 * bank:64 * bank + 64], t, 0, K, bb, t, 0, K)
        i, j = np.meshgrid(np.arange(64), np.arange(bank * half, bank * half + half), indexing="ij")
        lane, col = L.ws64_position(i, j, N)
        expect[lane, col] = ref[i, j]
    if not np.array_equal(got, expect):
        bad = np.argwhere(got != expect)[:6]
        raise AssertionError(f"{int((got != expect).sum())} cells differ; first {bad.tolist()}: "
                             f"got {[got[tuple(x)] for x in bad]} expect {[expect[tuple(x)] for x in bad]}")
