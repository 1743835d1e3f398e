"""Pins for the float64 GEMM oracle (CPU only).

Each pin ties the oracle to something other than itself: a library routine
(torch dtype decoding, numpy.matmul), a closed form (identity, permutation,
all-ones, power-of-two scales) or the worked example of the "tcgen05.mma"
page ("four K16 issues for a 128x64x64 product").  A planted-mistake test
shows the pins notice a transposed operand or a dropped scale.
"""
import numpy as np
import pytest
import torch

import synthetic as syn




# ---------------------------------------------------------------- decoders

def _torch_decode(bits, tdtype, itype):
    return torch.from_numpy(bits.astype(np.int64)).to(itype).view(tdtype).double().numpy()


def _same(a, b):
    nan = np.isnan(a)
    assert np.array_equal(nan, np.isnan(b))
    assert np.array_equal(a[~nan], b[~nan])


def test_decode_f16_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.float16).double().numpy()
    _same(oracle_mod.decode(bits, oracle_mod.F16), ref)


def test_decode_bf16_all_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    _same(oracle_mod.decode(bits, oracle_mod.BF16), ref)


def test_decode_e4m3_all_patterns(oracle_mod):
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).double().numpy()
    _same(oracle_mod.decode(bits, oracle_mod.E4M3), ref)


def test_decode_e8m0_all_patterns(oracle_mod):
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(torch.float8_e8m0fnu).double().numpy()
    _same(oracle_mod.decode_e8m0(bits), ref)


def test_decode_f32_sampled_and_special(oracle_mod):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 1, 0x007FFFFF, 0x00800000, 0x3F800000, 0x7F7FFFFF, 0x7F800000,
                        0x7FC00000, 0x80000000, 0x80000001, 0xFF800000], dtype=np.uint32)
    bits = np.concatenate([bits, special])
    ref = bits.view(np.float32).astype(np.float64)
    _same(oracle_mod.decode(bits, oracle_mod.F32), ref)


# ---------------------------------------------------------------- GEMM

def _logical(oracle_mod, A, a_type, a_major, B, b_type, b_major, M, N, K):
    """Decoded logical A (MxK) and B (KxN) via torch dtype views (library)."""
    tmap = {oracle_mod.F32: (np.uint32, None), oracle_mod.F16: (np.uint16, torch.float16),
            oracle_mod.BF16: (np.uint16, torch.bfloat16), oracle_mod.E4M3: (np.uint8, torch.float8_e4m3fn)}

    def dec(x, t):
        if t == oracle_mod.F32:
            return x.view(np.float32).astype(np.float64)
        npt, tt = tmap[t]
        if npt is np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(tt).double().numpy()
        return torch.from_numpy(x).view(tt).double().numpy()

    a = dec(A, a_type)
    b = dec(B, b_type)
    a = a if a_major == oracle_mod.K_MAJOR else a.T
    b = b.T if b_major == oracle_mod.K_MAJOR else b
    return a[:M, :K], b[:K, :N]


CASES = [
    ("bf16", "k", "k", 70, 90, 130),
    ("bf16", "k", "mn", 129, 64, 200),
    ("f16", "mn", "k", 33, 257, 96),
    ("f16", "mn", "mn", 1, 7, 48),
    ("tf32", "k", "k", 64, 40, 72),
    ("tf32", "mn", "mn", 17, 31, 33),
    ("e4m3", "k", "k", 40, 50, 128),
]
TYPE = {"f16": 1, "bf16": 2, "tf32": 0, "e4m3": 3}


@pytest.mark.parametrize("dtype,am,bm,M,N,K", CASES)
def test_gemm_matches_numpy_matmul(oracle_mod, dtype, am, bm, M, N, K):
    w = syn.Workload("t", M, N, K, dtype, am, bm, "uniform")
    x = syn.make_inputs(w)
    t = TYPE[dtype]
    ai = 0 if am == "k" else 1
    bi = 0 if bm == "k" else 1
    D, S = oracle_mod.gemm(M, N, K, x["A"], t, ai, x["lda"], x["B"], t, bi, x["ldb"])
    a, b = _logical(oracle_mod, x["A"], t, ai, x["B"], t, bi, M, N, K)
    np.testing.assert_allclose(D, a @ b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, np.abs(a) @ np.abs(b), rtol=1e-12, atol=1e-12)


def test_gemm_row_subset_matches_full(oracle_mod):
    w = syn.Workload("t", 50, 33, 70, "bf16", "k", "mn", "normal")
    x = syn.make_inputs(w)
    D, S = oracle_mod.gemm(50, 33, 70, x["A"], 2, 0, x["lda"], x["B"], 2, 1, x["ldb"])
    rows = [49, 0, 17, 17]
    Dr, Sr = oracle_mod.gemm(50, 33, 70, x["A"], 2, 0, x["lda"], x["B"], 2, 1, x["ldb"], rows=rows)
    assert np.array_equal(Dr, D[rows]) and np.array_equal(Sr, S[rows])


def test_gemm_identity_and_permutation_exact(oracle_mod):
    # A = I reproduces B bit for bit; A = P permutes B's rows.
    n = 64
    b = syn.draw((n, 96), 5, "uniform", n)
    B = syn.lay_out_b(syn.to_bits(b, "bf16"), "k")
    bdec = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).double().numpy().T
    I = syn.to_bits(np.eye(n), "bf16")
    D, _ = oracle_mod.gemm(n, 96, n, I, 2, 0, n, B, 2, 0, n)
    assert np.array_equal(D, bdec)
    perm = np.random.default_rng(3).permutation(n)
    P = syn.to_bits(np.eye(n)[perm], "bf16")
    D, _ = oracle_mod.gemm(n, 96, n, P, 2, 0, n, B, 2, 0, n)
    assert np.array_equal(D, bdec[perm])


def test_gemm_all_ones_gives_k(oracle_mod):
    M, N, K = 9, 11, 1000
    A = syn.to_bits(np.ones((M, K)), "f16")
    B = syn.to_bits(np.ones((N, K)), "f16")
    D, S = oracle_mod.gemm(M, N, K, A, 1, 0, K, B, 1, 0, K)
    assert np.all(D == K) and np.all(S == K)


def test_gemm_k_zero_gives_zero(oracle_mod):
    A = np.zeros((4, 0), np.uint16)
    B = np.zeros((5, 0), np.uint16)
    D, S = oracle_mod.gemm(4, 5, 0, A, 2, 0, 0, B, 2, 0, 0)
    assert np.all(D == 0) and np.all(S == 0)


def test_page_example_four_k16_issues_exact(oracle_mod):
    # "tcgen05.mma" page, example: a, b = integers(-4,5)/4 as float16 from
    # default_rng(0), a (128,64), b stored (N,K) = (64,64), checked against a @ b.T.
    rng = np.random.default_rng(0)
    a = (rng.integers(-4, 5, (128, 64)) / 4).astype("float16")
    b = (rng.integers(-4, 5, (64, 64)) / 4).astype("float16")
    D, _ = oracle_mod.gemm(128, 64, 64, a.view(np.uint16), 1, 0, 64, b.view(np.uint16), 1, 0, 64)
    ref = a.astype(np.float64) @ b.astype(np.float64).T
    assert np.array_equal(D, ref)  # quarter-integers: every partial sum is exact


def test_blockscaled_identity_closed_form(oracle_mod):
    # A = I (e4m3 1.0) with per-(row, K-block) exponents ea and B with exponents
    # eb: D[m,n] = 2^(ea[m, m//32] + eb[n, m//32] - 254) * e4m3(B)[m, n].
    n, N = 128, 40
    A = syn.to_bits(np.eye(n), "e4m3")
    b = syn.draw((n, N), 11, "normal1", n)
    B = syn.lay_out_b(syn.to_bits(b, "e4m3"), "k")
    rng = np.random.default_rng(12)
    SFA = (127 + rng.integers(-6, 7, size=(n, n // 32))).astype(np.uint8)
    SFB = (127 + rng.integers(-6, 7, size=(N, n // 32))).astype(np.uint8)
    D, _ = oracle_mod.gemm(n, N, n, A, 3, 0, n, B, 3, 0, n, SFA=SFA, SFB=SFB)
    bdec = torch.from_numpy(B).view(torch.float8_e4m3fn).double().numpy().T  # (K, N)
    m = np.arange(n)
    expo = SFA[m, m // 32].astype(np.int64)[:, None] + SFB[:, m // 32].T.astype(np.int64) - 254
    assert np.array_equal(D, np.ldexp(bdec, expo))


def test_blockscaled_matches_numpy(oracle_mod):
    w = syn.WORKLOADS["mxf8_8192"]
    x = syn.make_inputs(w, M=48, N=72, K=160)
    D, S = oracle_mod.gemm(48, 72, 160, x["A"], 3, 0, x["lda"], x["B"], 3, 0, x["ldb"],
                           SFA=x["SFA"], SFB=x["SFB"])
    a = torch.from_numpy(x["A"]).view(torch.float8_e4m3fn).double().numpy()
    b = torch.from_numpy(x["B"]).view(torch.float8_e4m3fn).double().numpy().T
    sa = np.repeat(np.ldexp(1.0, x["SFA"].astype(np.int64) - 127), 32, axis=1)[:, :160]
    sb = np.repeat(np.ldexp(1.0, x["SFB"].astype(np.int64) - 127), 32, axis=1)[:, :160].T
    ref = (a * sa) @ (b * sb)
    np.testing.assert_allclose(D, ref, rtol=1e-12, atol=0)
    np.testing.assert_allclose(S, np.abs(a * sa) @ np.abs(b * sb), rtol=1e-12)


def test_planted_mistakes_are_caught(oracle_mod):
    # Plant the mistakes a reader could make (transposed B, dropped scale) by
    # calling the oracle wrongly; the numpy pin must reject each one.
    w = syn.Workload("t", 24, 40, 64, "bf16", "k", "k", "uniform")
    x = syn.make_inputs(w)
    a, b = _logical(oracle_mod, x["A"], 2, 0, x["B"], 2, 0, 24, 40, 64)
    D_wrong_major, _ = oracle_mod.gemm(24, 40, 64, x["A"], 2, 0, x["lda"], x["B"], 2, 1, 40)
    assert not np.allclose(D_wrong_major, a @ b)
    wm = syn.WORKLOADS["mxf8_8192"]
    y = syn.make_inputs(wm, M=16, N=16, K=64)
    D_noscale, _ = oracle_mod.gemm(16, 16, 64, y["A"], 3, 0, 64, y["B"], 3, 0, 64, SFA=y["SFA"])
    D_full, _ = oracle_mod.gemm(16, 16, 64, y["A"], 3, 0, 64, y["B"], 3, 0, 64,
                                SFA=y["SFA"], SFB=y["SFB"])
    assert not np.allclose(D_noscale, D_full)


# ---------------------------------------------------------------------------
# E5M2 and the packed microscaling formats (E3M2, E2M3, E2M1)
# ---------------------------------------------------------------------------

def test_e5m2_decoder_matches_torch_over_all_codes(oracle_mod):
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    got = oracle_mod.decode(codes, oracle_mod.E5M2)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _embed(code, ebits, fbits, wide_ebits, wide_fbits, wide_bias, bias):
    """Bit fields of a normal narrow code re-based into a wider format's code
    (same sign and fraction, exponent shifted by the bias difference)."""
    s = (code >> (ebits + fbits)) & 1
    e = (code >> fbits) & ((1 << ebits) - 1)
    f = code & ((1 << fbits) - 1)
    return (s << 7) | ((e - bias + wide_bias) << wide_fbits) | (f << (wide_fbits - fbits))


@pytest.mark.parametrize("fmt,ebits,fbits,bias,wide", [
    ("E2M3", 2, 3, 1, "e4m3"), ("E3M2", 3, 2, 3, "e5m2"), ("E2M1", 2, 1, 1, "e4m3")])
def test_microscaling_normals_match_torch_8bit_decoders(oracle_mod, fmt, ebits, fbits, bias, wide):
    """Every normal E2M3 / E2M1 value is exactly an E4M3 value and every
    normal E3M2 value an E5M2 value (same fraction bits, exponent re-based):
    torch's 8-bit decoders give the expected values independently of the
    oracle's formula."""
    import torch
    bits = 1 + ebits + fbits
    all_codes = np.arange(1 << bits, dtype=np.uint8)
    normal = all_codes[((all_codes >> fbits) & ((1 << ebits) - 1)) != 0]
    wb, wf, wbias = (4, 3, 7) if wide == "e4m3" else (5, 2, 15)
    wide_codes = np.array([_embed(int(c), ebits, fbits, wb, wf, wbias, bias) for c in normal], dtype=np.uint8)
    tdt = torch.float8_e4m3fn if wide == "e4m3" else torch.float8_e5m2
    ref = torch.from_numpy(wide_codes).view(tdt).to(torch.float64).numpy()
    got = oracle_mod.decode(normal, getattr(oracle_mod, fmt))
    assert np.array_equal(got, ref), (fmt, got, ref)


def test_microscaling_constants_from_the_ocp_spec(oracle_mod):
    """The OCP Microscaling specification's tabulated limits: E2M3 max normal
    7.5, min normal 1.0, max subnormal 0.875, min subnormal 0.125; E3M2 28,
    0.25, 0.1875, 0.0625; E2M1 6, 1, 0.5 (its only subnormal); no infinities
    or NaNs, the sign in the top bit."""
    d = oracle_mod.decode
    for fmt, codes_vals in ((oracle_mod.E2M3, {0x1F: 7.5, 0x08: 1.0, 0x07: 0.875, 0x01: 0.125, 0x3F: -7.5}),
                            (oracle_mod.E3M2, {0x1F: 28.0, 0x04: 0.25, 0x03: 0.1875, 0x01: 0.0625, 0x3F: -28.0}),
                            (oracle_mod.E2M1, {0x7: 6.0, 0x2: 1.0, 0x1: 0.5, 0xF: -6.0})):
        for c, v in codes_vals.items():
            assert d(np.array([c], np.uint8), fmt)[0] == v, (fmt, hex(c))
    e2m1 = d(np.arange(16, dtype=np.uint8), oracle_mod.E2M1)
    assert e2m1.tolist()[:8] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(e2m1[8:], -e2m1[:8])
    for fmt, bits in ((oracle_mod.E2M3, 6), (oracle_mod.E3M2, 6), (oracle_mod.E2M1, 4)):
        v = d(np.arange(1 << bits, dtype=np.uint8), fmt)
        assert np.all(np.isfinite(v))
        pos = v[: 1 << (bits - 1)]
        assert np.all(np.diff(pos) > 0)  # codes 0 .. 2^(b-1)-1 are increasing magnitudes


def _bitstring_pack(codes_2d, bits):
    """Reference packer, one bit at a time: element j of a row at bits
    [bits*j, bits*(j+1)) of the row's little-endian bit string."""
    rows, n = codes_2d.shape
    out = np.zeros((rows, n * bits // 8), dtype=np.uint8)
    for r in range(rows):
        for j in range(n):
            for b in range(bits):
                if (int(codes_2d[r, j]) >> b) & 1:
                    pos = j * bits + b
                    out[r, pos // 8] |= np.uint8(1 << (pos % 8))
    return out


@pytest.mark.parametrize("fmt,bits,one", [("E2M3", 6, 0x08), ("E3M2", 6, 0x0C), ("E2M1", 4, 0x2)])
def test_packed_fetch_through_an_identity_gemm(oracle_mod, fmt, bits, one):
    """A (M x K codes, packed) times B = the K x K identity (code of 1.0 on the
    diagonal, scales 2^0) returns every decoded element of A at its (m, k):
    the oracle's packed-element fetch agrees with an independent bit-by-bit
    packer and with the input generator's packer; swapping the nibble or
    value order in the packing is caught."""
    import synthetic as syn
    M, K = 5, 64
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(M, K)).astype(np.uint8)
    A = _bitstring_pack(codes, bits)
    assert np.array_equal(A, syn.pack(codes, bits))
    eye = np.where(np.eye(K, dtype=bool), one, 0).astype(np.uint8)
    B = _bitstring_pack(eye, bits)
    t = getattr(oracle_mod, fmt)
    sfa = np.full((M, K // 32), 127, np.uint8)
    sfb = np.full((K, K // 32), 127, np.uint8)
    D, _ = oracle_mod.gemm(M, K, K, A, t, 0, K, B, t, 0, K, SFA=sfa, SFB=sfb)
    assert np.array_equal(D, oracle_mod.decode(codes, t))
    # planted mistake: the values of each pair (FP4) or group of four (FP6)
    # in reverse order
    g = 2 if bits == 4 else 4
    swapped = codes.reshape(M, K // g, g)[:, :, ::-1].reshape(M, K)
    D2, _ = oracle_mod.gemm(M, K, K, _bitstring_pack(swapped, bits), t, 0, K, B, t, 0, K, SFA=sfa, SFB=sfb)
    assert not np.array_equal(D2, D)


def test_ue4m3_scale_decoder_matches_torch(oracle_mod):
    """The NVFP4 scale is the E4M3FN encoding without a sign: codes 0..127
    decode as torch's float8_e4m3fn; codes with the top bit set are no scale."""
    import torch
    codes = np.arange(128, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle_mod.decode_ue4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])
    assert np.all(np.isnan(oracle_mod.decode_ue4m3(np.arange(128, 256, dtype=np.uint8))))


def test_block16_scales_identity_closed_form(oracle_mod):
    """A = I in E2M1 with one unsigned-E4M3 scale per 16 K elements: D[m, n]
    = sfa[m, m//16] * sfb[n, m//16] * B[n, m] exactly; a 32-wide block read
    (the MX rule) or an A/B scale swap is caught."""
    import synthetic as syn
    K, N = 64, 40
    A = syn.pack(np.where(np.eye(K, dtype=bool), 0x2, 0).astype(np.uint8), 4)
    codes = syn.codes((N, K), 77, 4)
    B = syn.pack(codes, 4)
    sfa = syn.ue4m3_scales(K, K, 78)
    sfb = syn.ue4m3_scales(N, K, 79)
    D, _ = oracle_mod.gemm(K, N, K, A, oracle_mod.E2M1, 0, K, B, oracle_mod.E2M1, 0, K, SFA=sfa, SFB=sfb,
                           sf_block=16, sf_kind=oracle_mod.SF_UE4M3)
    m = np.arange(K)
    expect = (oracle_mod.decode_ue4m3(sfa[m, m // 16])[:, None] * oracle_mod.decode_ue4m3(sfb[:, m // 16]).T
              * oracle_mod.decode(codes, oracle_mod.E2M1).T)
    assert np.array_equal(D, expect)
    # planted mistake: blocks of 32 read the wrong scale for half the rows
    sfa32 = sfa[:, ::2].copy()
    sfb32 = sfb[:, ::2].copy()
    D32, _ = oracle_mod.gemm(K, N, K, A, oracle_mod.E2M1, 0, K, B, oracle_mod.E2M1, 0, K, SFA=sfa32, SFB=sfb32,
                             sf_block=32, sf_kind=oracle_mod.SF_UE4M3)
    assert not np.array_equal(D32, D)


# ------------------------------------------------------------------ chained product

def test_encode_rne_bf16_matches_torch_rounding_of_fp32(oracle_mod):
    # torch rounds fp32 -> bf16 to nearest, ties to even; on fp32 inputs the
    # float64 encoder must agree bit for bit, including ties, subnormals and
    # values that round up into the next binade
    rng = np.random.default_rng(3)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(2.0) ** rng.integers(-20, 20, 20000)
    ties = (np.arange(0x3F800000, 0x3F800000 + 64 * 0x10000, 0x10000, dtype=np.uint64) + 0x8000).astype(np.uint32)
    special = np.array([0x3FFF8000, 0x3FFFFFFF, 0x00008000, 0x00018000, 0x007F8000, 0x80018000, 0x3F808000,
                        0x3F818000], dtype=np.uint32)
    x = np.concatenate([x, ties.view(np.float32), special.view(np.float32)])
    got = oracle_mod.encode_rne(x.astype(np.float64), oracle_mod.BF16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_encode_rne_closed_forms(oracle_mod):
    # halfway cases go to the even neighbour: bf16 has 8 significant bits,
    # f16 11 (1.0 = 0x3F80 / 0x3C00)
    bf = oracle_mod.encode_rne(np.array([1.0, 1 + 2 ** -7, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -9)]),
                               oracle_mod.BF16)
    assert bf.tolist() == [0x3F80, 0x3F81, 0x3F80, 0x3F82, 0xBF80]
    h = oracle_mod.encode_rne(np.array([1.0, 1 + 2 ** -10, 1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0]),
                              oracle_mod.F16)
    assert h.tolist() == [0x3C00, 0x3C01, 0x3C00, 0x3C02, 0x7BFF]


def _bits16(x, dtype):
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(dtype)
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_gemm_chain_small_integers_is_the_plain_product(oracle_mod, dt):
    # integers in [-2, 2] with K = 48: C is an integer of magnitude <= 192,
    # exact in both 16-bit types, so E = (A B1) B2 exactly
    rng = np.random.default_rng(5)
    M, N1, N2, K = 40, 32, 24, 48
    a, b1, b2 = (rng.integers(-2, 3, size=s).astype(np.float64) for s in ((M, K), (N1, K), (N2, N1)))
    tdt, odt = {"bf16": (torch.bfloat16, oracle_mod.BF16), "f16": (torch.float16, oracle_mod.F16)}[dt]
    E, S2, C, S1 = oracle_mod.gemm_chain(M, N1, N2, K, _bits16(a, tdt), _bits16(b1, tdt), _bits16(b2, tdt), odt)
    assert np.array_equal(C, a @ b1.T)
    assert np.array_equal(E, (a @ b1.T) @ b2.T)
    assert np.array_equal(S2, np.abs(a @ b1.T) @ np.abs(b2.T))
    assert np.array_equal(S1, np.abs(a) @ np.abs(b1.T))


def test_gemm_chain_rounds_the_intermediate(oracle_mod):
    # C = 1 + 2^-9 is not a bf16 number and rounds to 1 (f16 keeps it), so
    # E = B2 row sums scaled by the rounded C, not by the exact one
    M, N1, N2, K = 1, 16, 8, 2
    a = np.array([[1.0, 2 ** -9]])
    b1 = np.ones((N1, K))
    b2 = np.arange(N2 * N1, dtype=np.float64).reshape(N2, N1) / 16
    for tdt, odt, c in ((torch.bfloat16, oracle_mod.BF16, 1.0), (torch.float16, oracle_mod.F16, 1 + 2 ** -9)):
        E, _, C, _ = oracle_mod.gemm_chain(M, N1, N2, K, _bits16(a, tdt), _bits16(b1, tdt), _bits16(b2, tdt), odt)
        assert np.all(C == 1 + 2 ** -9)
        assert np.array_equal(E, np.full((1, N1), c) @ b2.T)


def test_gemm_chain_identity_second_factor_returns_the_rounded_intermediate(oracle_mod):
    rng = np.random.default_rng(9)
    M, N1, K = 30, 48, 200
    a = rng.standard_normal((M, K)).astype(np.float32)
    b1 = rng.standard_normal((N1, K)).astype(np.float32)
    eye = np.eye(N1, dtype=np.float32)
    E, _, C, _ = oracle_mod.gemm_chain(M, N1, N1, K, _bits16(a, torch.bfloat16), _bits16(b1, torch.bfloat16),
                                       _bits16(eye, torch.bfloat16), oracle_mod.BF16)
    rounded = torch.from_numpy(oracle_mod.encode_rne(C, oracle_mod.BF16).view(np.int16)).view(torch.bfloat16)
    assert np.array_equal(E, rounded.double().numpy())
