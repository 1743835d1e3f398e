"""Pins for the oracle's layout models (CPU only).

Pinned against: the pages' worked examples (the "tcgen05.cp" 128x128b copy of
arange(512) with (ldo=16, sdo=128, swizzle=0); the "tcgen05.mma" 128x64 fp16
K-major operand with (16, 1024, 3) and its K16 view rearrangement; the
"ldmatrix / stmatrix" interleaved-slots example), the CUDA driver header's
description of the TMA swizzle modes, the PTX mma.sync m16n8 accumulator
fragment (a textbook layout the 16x256b image must reduce to), and brute-force
bijection checks on every small case.
"""
import itertools

import numpy as np
import pytest

from oracle import layouts as L


# ------------------------------------------------------------ descriptor walk

def test_cp_walk_page_example_is_dense_row_major():
    # "tcgen05.cp" page example: shared (128, 4) uint32 written row-major from
    # arange(512), copied with (ldo=16, sdo=128, swizzle=0), read back equal.
    r, w = np.meshgrid(np.arange(128), np.arange(4), indexing="ij")
    off = L.cp_physical(0, r, w, 16, 128, 0)
    assert np.array_equal(off // 4, np.arange(512).reshape(128, 4))


def test_mma_page_example_operand_is_dense_and_k16_steps_are_32_bytes():
    # "tcgen05.mma" page example: fp16 (128, 64) K-major, descriptor (16, 1024, 3).
    m, k = np.meshgrid(np.arange(128), np.arange(64), indexing="ij")
    off = L.mma_operand_offset(m, k, 2, "k", 16, 1024, 3)
    assert np.array_equal(off, 128 * m + 2 * k)
    # The K16 repeat (view "m (kr k) -> kr m k") moves the origin by 32 bytes.
    for kr in range(4):
        k16 = np.arange(16)
        assert np.array_equal(L.mma_operand_offset(m[:, :16], 16 * kr + k16[None, :], 2, "k", 16, 1024, 3),
                              L.mma_operand_offset(m[:, :16], k16[None, :], 2, "k", 16, 1024, 3) + 32 * kr)


@pytest.mark.parametrize("s", [0, 1, 2, 3, 4])
def test_swizzle_is_a_period_closed_bijection(s):
    P = L.SWIZZLE_PERIOD[s] if s else 1024
    a = np.arange(4 * P)
    p = L.swizzle_addr(a, s)
    assert np.array_equal(np.sort(p), a)                      # bijection
    assert np.array_equal(L.swizzle_addr(p, s), a)            # involution
    assert np.array_equal(p[P:] - P, p[:-P])                  # period closure
    assert np.array_equal(p // L.SWIZZLE_PERIOD[s] if s else p // P, a // L.SWIZZLE_PERIOD[s] if s else a // P)


@pytest.mark.parametrize("s,span,gran", [(1, 32, 16), (2, 64, 16), (3, 128, 16), (4, 128, 32)])
def test_swizzle_matches_driver_header_description(s, span, gran):
    # cuda.h, CUtensorMapSwizzle: "Swizzle 16B chunks within 32B/64B/128B span"
    # and "Swizzle 32B chunks within 128B span" (the 128B_ATOM_32B mode).
    a = np.arange(8192)
    p = L.swizzle_addr(a, s)
    assert np.array_equal(p // span, a // span)                # stays in its span
    assert np.array_equal(p % gran, a % gran)                  # granules move whole
    # row 0 of every period is left in place
    per = L.SWIZZLE_PERIOD[s]
    first = (a % per) < span
    assert np.array_equal(p[first], a[first])


def test_swizzle_mode4_page_formula_on_example_offsets():
    # "swizzle=4": offset ^ ((offset >> 2) & 96): bytes 128..159 (K row 1,
    # first 32B granule) land in granule 1 of that row.
    assert L.swizzle_addr(128, 4) == 160
    assert L.swizzle_addr(256 + 96, 4) == 256 + 32
    assert L.swizzle_addr(384 + 64, 4) == 384 + 32  # row 3, granule 2 -> 2^3 = 1


def test_cp_walk_swizzled_words_contiguous_and_ldo_ignored():
    r, w = np.meshgrid(np.arange(16), np.arange(8), indexing="ij")
    for s in (1, 2, 3):
        a = L.cp_walk(r, w, 16, 1024, s)
        b = L.cp_walk(r, w, 4096, 1024, s)
        assert np.array_equal(a, b)
        assert np.array_equal(a - L.cp_walk(r, 0 * w, 16, 1024, s), 4 * w)


def test_descriptor_field_checks():
    L.check_descriptor(0, 16, 1024, 3)
    for bad in [(8, 16, 1024, 3), (0, 8, 1024, 3), (0, 16, 1 << 18, 3), (0, -16, 16, 0), (0, 16, 16, 5)]:
        with pytest.raises(ValueError):
            L.check_descriptor(*bad)


def test_mma_mn_major_unswizzled_swaps_strides():
    # MN-major unswizzled: row groups (of K) at LDO, contiguous 16-byte chunks at SDO.
    mn, k = np.meshgrid(np.arange(32), np.arange(16), indexing="ij")
    off = L.mma_operand_offset(mn, k, 2, "mn", 256, 4096, 0)
    assert np.array_equal(off, (k // 8) * 256 + (k % 8) * 16 + (mn // 8) * 4096 + (mn % 8) * 2)
    # and K-major unswizzled the other way round
    off = L.mma_operand_offset(mn, k, 2, "k", 256, 4096, 0)
    assert np.array_equal(off, (mn // 8) * 4096 + (mn % 8) * 16 + (k // 8) * 256 + (k % 8) * 2)


@pytest.mark.parametrize("eb,s,ldo", [(2, 3, 8192), (1, 3, 16384), (4, 4, 4096), (2, 1, 4096)])
def test_mma_mn_major_swizzled_tile_is_a_bijection(eb, s, ldo):
    rb = L.row_bytes(s)
    g = L.rows_per_group(s)
    mn_n = 2 * rb // eb
    k_n = 4 * g
    sdo = g * rb
    mn, k = np.meshgrid(np.arange(mn_n), np.arange(k_n), indexing="ij")
    off = L.mma_operand_offset(mn, k, eb, "mn", ldo, sdo, s)
    phys = L.swizzle_addr(off, s)
    vals = np.sort(phys.ravel())
    assert np.unique(vals // eb).size == mn_n * k_n


# ------------------------------------------------------------ TMEM ld/st images

@pytest.mark.parametrize("shape", L.LD_SHAPES)
@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
def test_ld_images_are_bijections(shape, n):
    if shape != "32x32b" and n > 64:
        pytest.skip("x128 only for 32x32b")
    regs = L.ld_regs_per_lane(shape, n)
    rows, cols = L.ld_atom_extent(shape, n)
    lanes = np.arange(32)[:, None]
    rr = np.arange(regs)[None, :]
    row, col = L.ld_owner(shape, lanes, rr)
    assert row.min() >= 0 and row.max() < rows and col.min() >= 0 and col.max() < cols
    assert np.unique(row * cols + col).size == rows * cols == 32 * regs


def test_ld_32x32b_is_lane_row_register_column():
    row, col = L.ld_owner("32x32b", np.arange(32)[:, None], np.arange(8)[None, :])
    assert np.array_equal(row, np.repeat(np.arange(32)[:, None], 8, 1))
    assert np.array_equal(col, np.repeat(np.arange(8)[None, :], 32, 0))


def test_ld_16x256b_x1_is_mma_m16n8_accumulator_fragment():
    # PTX ISA, mma.m16n8k16 f32 accumulator: groupID = lane>>2,
    # threadID_in_group = lane%4; c0,c1 at (groupID, 2*tig + {0,1}),
    # c2,c3 at (groupID + 8, 2*tig + {0,1}).
    for lane in range(32):
        g, t = lane >> 2, lane % 4
        expect = [(g, 2 * t), (g, 2 * t + 1), (g + 8, 2 * t), (g + 8, 2 * t + 1)]
        got = [tuple(int(v) for v in L.ld_owner("16x256b", lane, r)) for r in range(4)]
        assert got == expect


def test_layout_b_roundtrip_positions_cover_tmem():
    i, j = np.meshgrid(np.arange(64), np.arange(128), indexing="ij")
    lane, col = L.layout_b_position(i, j)
    assert np.unique(lane * 64 + col).size == 128 * 64
    # the page's explicit register layout: [i, j] -> thread i + 64*(j//64), slot j%64
    assert np.array_equal(lane, i + 64 * (j // 64)) and np.array_equal(col, j % 64)


# ------------------------------------------------------------ ldmatrix

def test_ldmatrix_page_example_interleaved_slots():
    # "ldmatrix / stmatrix" page example: x (16,4,2) = arange(128); shared
    # layout (16,4,2):(8,1,128); S_std[k,m,r,w] = SM[2r+m, w, k]; two x2
    # issues (k = 0, 1) into register slots {0, 2} and {8, 10}; every other
    # slot keeps the sentinel 4294966519.
    x = np.arange(128, dtype=np.uint64).reshape(16, 4, 2)
    out = np.full((32, 12), 4294966519, dtype=np.uint64)
    for k in range(2):
        rows = [[[int(x[2 * r + m, w, k]) for w in range(4)] for r in range(8)] for m in range(2)]
        regs = L.ldmatrix_load(rows, 2)
        for lane in range(32):
            for m in range(2):
                # each b32 word is whole here (values < 2^16 sit in the low half)
                out[lane, 8 * k + 2 * m] = regs[lane][m]
    # expected array exactly as the page prints it
    expected = np.full((32, 12), 4294966519, dtype=np.uint64)
    for lane in range(32):
        for k in range(2):
            for matrix in range(2):
                expected[lane, 8 * k + 2 * matrix] = x[2 * (lane // 4) + matrix, lane % 4, k]
    assert np.array_equal(out, expected)


def test_ldmatrix_address_providers_and_trans():
    assert [L.ldmatrix_address_provider(m, r) for m in range(4) for r in range(8)] == list(range(32))
    # .trans: register element (row, 2w+h) comes from shared element (2w+h, row)
    rows = [[[((2 * w) + 16 * r) | (((2 * w + 1) + 16 * r) << 16) for w in range(4)] for r in range(8)]]
    regs = L.ldmatrix_load(rows, 1, trans=True)  # shared element (r, c) holds 16r + c
    for lane in range(32):
        row, w = lane // 4, lane % 4
        lo, hi = regs[lane][0] & 0xFFFF, regs[lane][0] >> 16
        assert lo == 16 * (2 * w) + row and hi == 16 * (2 * w + 1) + row


def test_stmatrix_inverts_ldmatrix():
    # "Transpose and stores": stmatrix takes the load's register image as input
    # and writes each provider's row, so a store followed by a load (same count,
    # same .trans) returns the registers, and a load then a store the rows.
    rng = np.random.default_rng(11)
    for count in (1, 2, 4):
        for trans in (False, True):
            regs = [[int(v) for v in rng.integers(0, 2**32, size=count, dtype=np.uint64)] for _ in range(32)]
            rows = L.stmatrix_store(regs, count, trans)
            assert L.ldmatrix_load(rows, count, trans) == regs
            rows2 = [[[int(v) for v in rng.integers(0, 2**32, size=4, dtype=np.uint64)] for _ in range(8)]
                     for _ in range(count)]
            assert L.stmatrix_store(L.ldmatrix_load(rows2, count, trans), count, trans) == rows2


def test_stmatrix_owners_and_trans_direct():
    # non-transposed: row r word w of matrix m comes whole from lane 4r + w's
    # m-th register ("Register word (matrix,row,word) belongs to lane 4*row+word")
    regs = [[1000 * lane + m for m in range(4)] for lane in range(32)]
    rows = L.stmatrix_store(regs, 4)
    for m, r, w in itertools.product(range(4), range(8), range(4)):
        assert rows[m][r][w] == 1000 * (4 * r + w) + m
    # .trans of 16-bit elements: register element (i, j) = 16i + j (lane 4i + j//2,
    # half j%2) lands at shared element (j, i)
    regs = [[(16 * (lane // 4) + 2 * (lane % 4)) | ((16 * (lane // 4) + 2 * (lane % 4) + 1) << 16)]
            for lane in range(32)]
    rows = L.stmatrix_store(regs, 1, trans=True)
    for r, c in itertools.product(range(8), range(8)):
        assert (rows[0][r][c // 2] >> (16 * (c % 2))) & 0xFFFF == 16 * c + r


# ------------------------------------------------------------ split accesses

SPLIT_IMMS = [(16, 8), (16, 0), (0, 16), (16, 16)]


def test_split_page_example_quadrants():
    # "Split accesses: 16x32bx2" example: .x4 with imm_half_splitoff (16 << 16) + 8
    # reads mem[:, :16, :4] for the first access and mem[:, 16:32, 8:12] for the second
    row, col = L.split_owner(np.arange(32)[:, None], np.arange(4)[None, :], 16, 8)
    assert set(zip(row[:16].ravel(), col[:16].ravel())) == {(i, j) for i in range(16) for j in range(4)}
    assert set(zip(row[16:].ravel(), col[16:].ravel())) == {(i, j) for i in range(16, 32) for j in range(8, 12)}
    # lane l owns (access l//16, row l%16, column r)
    assert np.array_equal(row, np.arange(32)[:, None] % 16 + 16 * (np.arange(32)[:, None] // 16) + 0 * col)
    assert np.array_equal(col, np.arange(4)[None, :] + 8 * (np.arange(32)[:, None] // 16))


def test_split_with_sixteen_lane_offset_is_the_32_lane_shape():
    # immediate (16 << 16) + 0: the two 16-lane accesses stack into the 32x32b image
    for num in (1, 2, 4, 8):
        lanes, regs = np.arange(32)[:, None], np.arange(num)[None, :]
        assert all(np.array_equal(a, b) for a, b in
                   zip(L.split_owner(lanes, regs, 16, 0), L.ld_owner("32x32b", lanes, regs)))


def test_split_store_inverts_split_load():
    rng = np.random.default_rng(5)
    for (il, ic), num in itertools.product(SPLIT_IMMS, (1, 2, 4, 8)):
        regs = rng.integers(1, 2**32, size=(32, num), dtype=np.uint64)
        img = L.split_store(regs, il, ic)
        assert np.count_nonzero(img) == 32 * num
        assert np.array_equal(L.split_load(num, il, ic, lambda r, c: img[r, c]), regs)
    with pytest.raises(ValueError):
        L.split_store(np.ones((32, 4), dtype=np.uint64), 0, 2)  # second access overlaps the first


# ------------------------------------------------------------ scale factors

def test_sf_chunk_offset_through_cp_warpx4_lands_where_mma_reads():
    # "tcgen05.cp" table (32x128b.warpx4: 32 lanes, four replicas 32 apart) composed
    # with the chunk offset must give the "tcgen05.mma" block-scale placement
    # (lane r%32, byte-column 4*(r//32)+sf, four replicas).
    for r, kb in itertools.product(range(128), range(4)):
        off = int(L.sf_chunk_offset(r, kb))
        lanes_cp, col_cp, byte_cp = L.cp_32x128b_warpx4_position(off // 16, off % 16)
        lanes_sf, col_sf, byte_sf = L.sf_tmem_position(r, kb)
        assert np.array_equal(lanes_cp, lanes_sf) and col_cp == col_sf and byte_cp == byte_sf


def test_sf_chunk_offsets_fill_one_chunk_once():
    r, kb = np.meshgrid(np.arange(128), np.arange(4), indexing="ij")
    off = L.sf_chunk_offset(r, kb)
    assert np.array_equal(np.sort(off.ravel()), np.arange(512))


@pytest.mark.parametrize("rows,kblocks,tile_rows", [(128, 4, 128), (300, 9, 128), (256, 8, 256), (500, 5, 224)])
def test_sf_prepare_is_invertible(rows, kblocks, tile_rows):
    rng = np.random.default_rng(rows)
    sf = rng.integers(0, 255, size=(rows, kblocks)).astype(np.uint8)
    img = L.sf_prepare(sf, rows, kblocks, tile_rows)
    for r in range(rows):
        t, rl = divmod(r, tile_rows)
        c, rc = divmod(rl, 128)
        for kk in range(kblocks):
            ks, kb = divmod(kk, 4)
            assert img[ks, t, c, int(L.sf_chunk_offset(rc, kb))] == sf[r, kk]


# ------------------------------------------------------------- cp decompression

def _pack_bits(values, bits, rng):
    """Independent packer: set the block's bits one by one (value i at bit
    offsets bits*i .. bits*i + bits - 1, little-endian over the 16 bytes),
    then fill the padding bytes with random data."""
    block = bytearray(16)
    for i, v in enumerate(values):
        for b in range(bits):
            if (v >> b) & 1:
                pos = bits * i + b
                block[pos // 8] |= 1 << (pos % 8)
    data_bytes = 2 * bits  # 16 values x bits / 8
    block[data_bytes:] = bytes(rng.integers(0, 256, 16 - data_bytes, dtype=np.uint8))
    return np.frombuffer(bytes(block), dtype="<u4").copy()


def test_cp_decompress_fp4_nibble_sequence():
    # data bytes 0x10 0x32 ... 0xFE hold the nibbles 0, 1, ..., 15 in order;
    # each gains two low zero bits, so byte i is 4 * i
    block = np.array([0x76543210, 0xFEDCBA98, 0xDEADBEEF, 0x01234567], dtype=np.uint32)
    out = L.cp_decompress(block, 4)
    assert np.frombuffer(out.astype("<u4").tobytes(), dtype=np.uint8).tolist() == [4 * i for i in range(16)]


@pytest.mark.parametrize("fmt", [4, 6])
def test_cp_decompress_matches_bitwise_packer_and_ignores_padding(fmt):
    rng = np.random.default_rng(fmt)
    for _ in range(200):
        vals = rng.integers(0, 1 << fmt, 16)
        block = _pack_bits(vals, fmt, rng)
        other = block.copy()
        other[3] ^= 0xA5A5A5A5 if fmt == 4 else 0  # FP4 padding is all of word 3 (and word 2)
        if fmt == 4:
            other[2] ^= 0x5A5A5A5A
        got = np.frombuffer(L.cp_decompress(block, fmt).astype("<u4").tobytes(), dtype=np.uint8)
        exp = (vals << 2) if fmt == 4 else vals
        assert got.tolist() == exp.tolist()
        assert np.array_equal(L.cp_decompress(other, fmt), L.cp_decompress(block, fmt))
        assert np.all(got >> 6 == 0)            # two high zero bits either way
        if fmt == 4:
            assert np.all(got & 3 == 0)         # FP4: two low zero bits


def test_cp_decompress_fp6_padding_is_the_last_word():
    rng = np.random.default_rng(9)
    vals = rng.integers(0, 64, (5, 16))
    blocks = np.stack([_pack_bits(v, 6, rng) for v in vals])
    flipped = blocks.copy()
    flipped[:, 3] ^= 0xFFFFFFFF
    assert np.array_equal(L.cp_decompress(blocks, 6), L.cp_decompress(flipped, 6))
    flipped = blocks.copy()
    flipped[:, 2] ^= 1 << 31  # bit 95: the top bit of value 15
    diff = L.cp_decompress(flipped, 6) != L.cp_decompress(blocks, 6)
    assert diff[:, 3].all() and not diff[:, :3].any()


# ---------------------------------------------------------------------------
# The operand images the MMA image probe feeds to the hardware: every case is
# a bijection into its image, and each case tells the pages' assignment of
# LDO and SDO apart from the swapped one, so that the GPU comparison pins the
# model's stride roles (not only its shape).
# ---------------------------------------------------------------------------

def test_mma_image_cases_are_injective_and_discriminating():
    import sys, os
    sys.path.insert(0, os.path.dirname(__file__))
    from mma_image_cases import CASES, element_addresses, build_image, kstep

    for c in CASES:
        ks = c.K // kstep(c.dtype)
        for spec, rows in ((c.a, 128), (c.b, c.N)):
            bits = np.arange(rows * c.K, dtype=np.uint32).reshape(rows, c.K) + 1
            if c.dtype != "tf32":
                bits = bits.astype(np.uint16)
            img = build_image(bits, spec, c.dtype, ks)
            assert img.size <= 96 * 1024, c.name
            addr = element_addresses(spec, rows, c.dtype, ks)
            swapped = element_addresses(spec, rows, c.dtype, ks, ldo=spec.sdo, sdo=spec.ldo)
            moved = addr != swapped
            if spec.major == "k" and spec.swizzle != 0:
                # swizzled K-major ignores LDO (atoms fit in one row): the
                # swapped reading differs through SDO alone
                assert moved.any() or spec.ldo == spec.sdo, c.name
            else:
                assert moved.any(), f"{c.name}: strides indistinguishable"


def test_mma_operand_offset_mn_major_examples():
    """Closed-form values of the MN-major walk, worked out from the page's
    table: swizzled rows enumerate K (SDO between 8-row groups), contiguous
    chunks of one row width along M/N are LDO apart; unswizzled the roles swap
    (16-byte rows, LDO between 8-row groups of K, SDO between 8-element M/N
    chunks); mode 4 groups four 128-byte K rows per SDO."""
    # bf16, mode 3 (128-byte rows of 64 elements)
    assert L.mma_operand_offset(0, 0, 2, "mn", 8192, 1024, 3) == 0
    assert L.mma_operand_offset(63, 0, 2, "mn", 8192, 1024, 3) == 126
    assert L.mma_operand_offset(64, 0, 2, "mn", 8192, 1024, 3) == 8192
    assert L.mma_operand_offset(0, 7, 2, "mn", 8192, 1024, 3) == 7 * 128
    assert L.mma_operand_offset(0, 8, 2, "mn", 8192, 1024, 3) == 1024
    # bf16, mode 0: element (mn, k) in the 8x8 core block (k//8, mn//8)
    assert L.mma_operand_offset(9, 3, 2, "mn", 128, 1024, 0) == 1 * 1024 + 3 * 16 + 2
    assert L.mma_operand_offset(9, 11, 2, "mn", 128, 1024, 0) == 1 * 128 + 1 * 1024 + 3 * 16 + 2
    # tf32, mode 4: 32 elements per 128-byte row, 4 K rows per 512-byte group
    assert L.mma_operand_offset(33, 5, 4, "mn", 4096, 512, 4) == 4096 + 1 * 512 + 1 * 128 + 4
    # K-major, mode 0: 8-row groups SDO apart, 16-byte K chunks LDO apart
    assert L.mma_operand_offset(10, 9, 2, "k", 2048, 128, 0) == 1 * 128 + 2 * 16 + 1 * 2048 + 2


# ---------------------------------------------------------------------------
# Descriptor rules that depend on the allocation ("tcgen05.cp" page, "Shared
# descriptor address walk", second paragraph; "tcgen05.mma" page, "Shared
# descriptors are byte-stride contracts", last paragraph).  Each case is one
# sentence of the pages turned into an accepted and a rejected example.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("s,period", [(1, 256), (2, 512), (3, 1024), (4, 512)])
def test_swizzled_bases_need_period_alignment(s, period):
    # "Swizzled bases require 256/512/1024-byte period alignment for modes
    # 1/2/3"; mode 4 has "a 512-byte period" and backing allocations "align to
    # the full swizzle period".
    L.check_base(period, s)
    L.check_base(3 * period, s)
    for bad in (period // 2, period + 16, 128 if period > 128 else 16):
        with pytest.raises(ValueError, match="period"):
            L.check_base(bad, s)
    L.check_base(16, 0)  # unswizzled: any 16-byte aligned base


def test_walk_origin_swizzle_phase_decides_the_physical_bytes():
    # "The complete physical walk is checked, including the origin's swizzle
    # phase": 16 bytes from origin 512 of a mode-3 allocation are logically
    # bytes 512..527, inside a 576-byte backing, but the origin sits in row 4
    # of its 1024-byte period, so the 16-byte chunk moves to 576..591.
    with pytest.raises(ValueError, match="physical"):
        L.check_walk(512, 1, 4, 16, 1024, 3, base=0, backing=576)
    phys = L.check_walk(512, 1, 4, 16, 1024, 3, base=0, backing=None)
    assert phys.ravel().tolist() == [576, 580, 584, 588]
    # the same walk at phase 0 stays where it is
    assert L.check_walk(0, 1, 4, 16, 1024, 3, base=0, backing=1024).ravel().tolist() == [0, 4, 8, 12]
    # the phase is the absolute address's: a period-aligned base changes nothing
    assert np.array_equal(L.check_walk(512, 1, 4, 16, 1024, 3, base=4096), phys)


def test_four_row_region_needs_eight_row_backing():
    # "A 4-row logical region still needs a backing storage block large enough
    # for the descriptor's eight-row organization".  4 x 256b (4 rows, 8 words)
    # unswizzled with LDO 128: the words touched end at byte 192, but the two
    # 16-byte columns each belong to an 8-row block of 128 bytes.
    phys = L.check_walk(0, 4, 8, 128, 256, 0, backing=1 << 20)
    assert phys.max() + 4 == 192
    with pytest.raises(ValueError, match="eight-row"):
        L.check_walk(0, 4, 8, 128, 256, 0, backing=192)
    L.check_walk(0, 4, 8, 128, 256, 0, backing=256)
    # swizzled 128-byte rows: 4 rows use 512 bytes, the organisation 1024
    with pytest.raises(ValueError, match="eight-row"):
        L.check_walk(0, 4, 4, 16, 1024, 3, backing=512)
    L.check_walk(0, 4, 4, 16, 1024, 3, backing=1024)


def test_walk_rules_planted_mistakes_are_caught():
    # a wrong period (mode 2 taken as 256 bytes) or a walk checked on logical
    # instead of physical addresses would each let one of these through
    with pytest.raises(ValueError, match="period"):
        L.check_walk(0, 8, 4, 16, 512, 2, base=256, backing=4096)
    with pytest.raises(ValueError, match="physical"):
        L.check_walk(512 + 32, 1, 4, 16, 1024, 3, base=0, backing=512 + 64)


def test_gpu_cp_probe_cases_obey_the_walk_rules():
    # every tcgen05.cp case the GPU probe runs is a legal walk of its image
    import test_gpu_probes as g
    rows = {0: 128, 1: 128, 2: 32, 3: 4}
    words = {0: 8, 1: 4, 2: 4, 3: 8}
    for shape, origin, ldo, sdo, sw, nwords in g.CP_CASES + g.DECOMP_CASES:
        L.check_walk(origin, rows[shape % 4], words[shape % 4], ldo, sdo, sw, base=0, backing=4 * nwords)


@pytest.mark.parametrize("N", [64, 128, 256])
def test_ws64_layout_is_a_bijection_and_is_layout_b_at_n128(N):
    i, j = np.meshgrid(np.arange(64), np.arange(N), indexing="ij")
    lane, col = L.ws64_position(i, j, N)
    cells = lane * (N // 2) + col
    assert np.array_equal(np.sort(cells.ravel()), np.arange(64 * N))   # 128 lanes x N/2 columns, once each
    if N == 128:  # the "tcgen05.ld / tcgen05.st" page's Layout B formula
        lb, cb = L.layout_b_position(i, j)
        assert np.array_equal(lane, lb) and np.array_equal(col, cb)
