"""Layout models from the Apache TVM TIRx tcgen05 / ldmatrix documentation pages.

TEST INFRASTRUCTURE ONLY: used by the tests to predict, bit for bit, what the
GPU layout probes must return.  Shares nothing with the CUDA library.

Every function cites the page and section it restates.  Readings of points the
pages leave open are marked READING in the function that takes them (the XOR
of swizzle modes 1-3, the 16x64b register formula as printed, the packing
order inside an FP4 / FP6 decompression block); each is pinned bit for bit by
a GPU layout probe.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Swizzle modes ("tcgen05.cp" page, "Shared descriptor address walk";
# "tcgen05.mma" page, "Shared descriptors are byte-stride contracts" and
# "swizzle=4").
# ---------------------------------------------------------------------------

#: swizzle period in bytes for the pages' logical modes 0..4
SWIZZLE_PERIOD = {0: 16, 1: 256, 2: 512, 3: 1024, 4: 512}


def row_bytes(swizzle: int) -> int:
    """A descriptor row is ``16 << swizzle`` bytes for modes 0..3 and 128 bytes
    for mode 4 (128-byte span)."""
    return 128 if swizzle == 4 else (16 << swizzle)


def rows_per_group(swizzle: int) -> int:
    """Modes 0..3 group eight rows per SDO; mode 4 groups four K rows."""
    return 4 if swizzle == 4 else 8


def swizzle_addr(addr, swizzle: int):
    """Physical shared byte address for a logical one.

    Mode 4 is the page's formula ``offset ^ ((offset >> 2) & 96)``.
    READING (modes 1..3, the pages give only their 256/512/1024-byte periods):
    the 16-byte chunk index (address bits 4..3+s) is XORed with the s address
    bits starting at bit 7, i.e. ``addr ^ ((addr >> 3) & (((1 << s) - 1) << 4))``,
    applied to the absolute address; this is what makes the period alignment
    of swizzled bases and the origin's swizzle phase matter.
    Works elementwise on numpy integer arrays.
    """
    if swizzle == 0:
        return addr
    if swizzle == 4:
        return addr ^ ((addr >> 2) & 96)
    mask = ((1 << swizzle) - 1) << 4
    return addr ^ ((addr >> 3) & mask)


def cp_walk(r, w, ldo: int, sdo: int, swizzle: int):
    """Logical byte offset of (row r, b32 word w) of a tcgen05.cp source image
    relative to the descriptor origin ("tcgen05.cp" page, "Shared descriptor
    address walk"): row r starts at (r//8)*SDO + (r%8)*(16<<swizzle); without
    swizzle word w adds (w//4)*LDO + (w%4)*4; with swizzle words are contiguous
    and add 4*w (LDO ignored)."""
    r = np.asarray(r)
    w = np.asarray(w)
    base = (r // 8) * sdo + (r % 8) * (16 << swizzle)
    if swizzle == 0:
        return base + (w // 4) * ldo + (w % 4) * 4
    return base + 4 * w


def check_descriptor(origin: int, ldo: int, sdo: int, swizzle: int) -> None:
    """Field constraints ("tcgen05.cp" page, "Shared descriptor address walk";
    "tcgen05.mma" page, descriptor contract): strides are non-negative 16-byte
    multiples below 2^18, origins 16-byte aligned, the mode one of 0..4.
    Raises ValueError.  The rules that depend on the allocation (period
    alignment, the physical walk, eight-row backing) are :func:`check_walk`'s."""
    for name, v in (("ldo", ldo), ("sdo", sdo)):
        if v < 0 or v % 16 or v >= (1 << 18):
            raise ValueError(f"{name}={v} must be a non-negative multiple of 16 below 2^18")
    if origin % 16:
        raise ValueError(f"origin {origin} is not 16-byte aligned")
    if swizzle not in (0, 1, 2, 3, 4):
        raise ValueError(f"swizzle mode {swizzle} not in 0..4")


def check_base(base: int, swizzle: int) -> None:
    """"period": an allocation read through a swizzled descriptor starts on
    its mode's period, 256 / 512 / 1024 bytes for modes 1 / 2 / 3 ("tcgen05.cp"
    page, "Shared descriptor address walk") and 512 for mode 4 ("tcgen05.mma"
    page, "swizzle=4"; its backing allocations align to the full period).
    Raises ValueError."""
    if swizzle and base % SWIZZLE_PERIOD[swizzle]:
        raise ValueError(f"period: base {base} is not aligned to the {SWIZZLE_PERIOD[swizzle]}-byte period of "
                         f"mode {swizzle}")


def check_walk(origin: int, rows: int, words: int, ldo: int, sdo: int, swizzle: int,
               base: int = 0, backing: int | None = None):
    """The descriptor rules of the "tcgen05.cp" page ("Shared descriptor
    address walk") and the "tcgen05.mma" page's descriptor contract, applied
    to a walk of ``rows`` rows x ``words`` b32 words from ``origin`` bytes into
    an allocation that starts at shared byte address ``base`` and holds
    ``backing`` bytes (None: unbounded).  Raises ValueError naming the rule
    broken, in this order:

    * the field constraints of :func:`check_descriptor`;
    * "period": a swizzled allocation must start on its mode's period (256,
      512, 1024 bytes for modes 1, 2, 3; 512 for mode 4);
    * "physical": the complete physical walk, i.e. the swizzle applied to the
      absolute address base + origin + walk (so the origin's position inside
      its swizzle period, its phase, decides where each word lands), must stay
      inside the backing;
    * "eight-row": every row group the walk touches must be backed whole, as
      the descriptor organises rows in groups of eight even when fewer are
      used -- READING: for swizzled modes the group is 8 rows of 16 << mode
      bytes from the group's first row; unswizzled it is the 8 x 16-byte block
      of each 16-byte column the walk reads (LDO apart).

    Returns the physical byte address of every word, shape (rows, words),
    relative to ``base``."""
    check_descriptor(origin, ldo, sdo, swizzle)
    check_base(base, swizzle)
    if swizzle == 4:
        raise ValueError("mode 4 is an MMA operand mode; tcgen05.cp walks use modes 0..3")
    r, w = np.meshgrid(np.arange(rows), np.arange(words), indexing="ij")
    phys = swizzle_addr(base + origin + cp_walk(r, w, ldo, sdo, swizzle), swizzle) - base
    if backing is None:
        return phys
    if phys.min() < 0 or phys.max() + 4 > backing:
        raise ValueError(f"physical: the walk reaches bytes [{phys.min()}, {phys.max() + 4}) outside the "
                         f"{backing}-byte backing")
    rb = row_bytes(swizzle)
    if swizzle == 0:
        columns = [j * ldo for j in range(-(-words // 4))]
        block = 8 * 16
    else:
        columns = [0]
        block = 8 * rb
    for g in range(-(-rows // 8)):
        for c in columns:
            lo = origin + g * sdo + c
            chunk = swizzle_addr(base + np.arange(lo, lo + block, 16), swizzle) - base
            if chunk.min() < 0 or chunk.max() + 16 > backing:
                raise ValueError(f"eight-row: row group {g} occupies bytes up to {chunk.max() + 16}, beyond the "
                                 f"{backing}-byte backing")
    return phys


def cp_physical(origin: int, r, w, ldo: int, sdo: int, swizzle: int, base_align: int = 0):
    """Physical byte address (relative to a period-aligned allocation) of word
    (r, w) read by tcgen05.cp: the selected swizzle of origin + walk.  The
    origin is given un-swizzled ("tcgen05.mma" page: the origin is
    inverse-swizzled before encoding so it is not permuted twice; the swizzles
    are involutions, so the un-swizzled origin is what the descriptor holds)."""
    check_descriptor(origin, ldo, sdo, swizzle)
    return swizzle_addr(base_align + origin + cp_walk(r, w, ldo, sdo, swizzle), swizzle) - base_align


def cp_decompress(words, fmt: int):
    """FP4 / FP6 decompression of tcgen05.cp ("tcgen05.cp" page, "Native
    FP4/FP6 decompression").  ``words`` is an array (..., 4) of b32 words, one
    16-byte source block per row of the last axis: sixteen packed values
    followed by padding (FP4, fmt 4: 8 data bytes + 8 padding bytes; FP6,
    fmt 6: 12 data bytes + 4 padding bytes).  The destination block is sixteen
    bytes, value i in byte i; a 4-bit value gains two low zero bits
    (byte = v << 2), a 6-bit value two high zero bits (byte = v).
    READING (the page does not state the packing order): little-endian,
    value i occupies bits [b*i, b*(i+1)) of the data bytes read as one
    little-endian integer (b = 4 or 6).  Returns the (..., 4) destination
    words (little-endian bytes)."""
    w = np.asarray(words, dtype=np.uint64)
    if w.shape[-1] != 4:
        raise ValueError("blocks are 4 words")
    if fmt not in (4, 6):
        raise ValueError("fmt is 4 (FP4) or 6 (FP6)")
    mask = (1 << fmt) - 1
    flat = w.reshape(-1, 4)
    out = np.zeros(flat.shape, dtype=np.uint32)
    for n, blk in enumerate(flat):
        data = sum(int(blk[j]) << (32 * j) for j in range(4))  # the block as a 128-bit integer
        dst = 0
        for i in range(16):
            v = (data >> (fmt * i)) & mask
            dst |= ((v << 2) if fmt == 4 else v) << (8 * i)
        for j in range(4):
            out[n, j] = (dst >> (32 * j)) & 0xFFFFFFFF
    return out.reshape(w.shape)


def mma_operand_offset(mn, k, elem_bytes: int, major: str, ldo: int, sdo: int, swizzle: int):
    """Logical byte offset of operand element (mn, k) of a tcgen05.mma shared
    operand ("tcgen05.mma" page, "Shared descriptors are byte-stride
    contracts" and "swizzle=4").

    K-major: rows enumerate M/N, a row holds contiguous K elements; the next
    row group (8 rows) is SDO away and the next 16-byte chunk (unswizzled) LDO
    away; swizzled instruction atoms fit within one row.
    MN-major swizzled: rows enumerate K; row group stride SDO; the next
    contiguous M/N chunk (one row width) is LDO away.
    MN-major unswizzled: the two strides swap (LDO for row groups, SDO for
    chunks).
    Mode 4 (32-bit MN-major only): four K rows of 128 bytes per SDO, LDO to the
    next 128-byte M/N chunk.
    """
    mn = np.asarray(mn)
    k = np.asarray(k)
    rb = row_bytes(swizzle)
    g = rows_per_group(swizzle)
    if major == "k":
        byte = k * elem_bytes
        if swizzle == 0:
            return (mn // 8) * sdo + (mn % 8) * 16 + (byte // 16) * ldo + byte % 16
        if np.any(byte >= rb):
            raise ValueError("a K-major swizzled atom must fit within one row")
        return (mn // g) * sdo + (mn % g) * rb + byte
    if major == "mn":
        byte = mn * elem_bytes
        if swizzle == 0:
            return (k // 8) * ldo + (k % 8) * 16 + (byte // 16) * sdo + byte % 16
        return (k // g) * sdo + (k % g) * rb + (byte // rb) * ldo + byte % rb
    raise ValueError(major)


# ---------------------------------------------------------------------------
# tcgen05.ld / tcgen05.st register images ("tcgen05.ld / tcgen05.st" page,
# "Native images").
# ---------------------------------------------------------------------------

LD_SHAPES = ("32x32b", "16x64b", "16x128b", "16x256b")


def ld_regs_per_lane(shape: str, n: int) -> int:
    return {"32x32b": n, "16x64b": n, "16x128b": 2 * n, "16x256b": 4 * n}[shape]


def ld_atom_extent(shape: str, n: int):
    return {"32x32b": (32, n), "16x64b": (16, 2 * n), "16x128b": (16, 4 * n),
            "16x256b": (16, 8 * n)}[shape]


def ld_owner(shape: str, lane, reg):
    """(row, column) of the atom held in register ``reg`` of lane ``lane``.

    32x32b:  (l, r)
    16x64b:  (l//4 + 8(l%2), l//2%2 + 2r)        READING: as printed
    16x128b: (l//4 + 8(r%2), l%4 + 4(r//2))
    16x256b: (l//4 + 8(r//2%2), r%2 + 2(l%4) + 8(r//4))
    (The garbled "8(x)" of the page is 8*(x).)
    """
    l = np.asarray(lane)
    r = np.asarray(reg)
    if shape == "32x32b":
        row, col = l + 0 * r, r + 0 * l
    elif shape == "16x64b":
        row, col = l // 4 + 8 * (l % 2) + 0 * r, (l // 2) % 2 + 2 * r
    elif shape == "16x128b":
        row, col = l // 4 + 8 * (r % 2), l % 4 + 4 * (r // 2)
    elif shape == "16x256b":
        row, col = l // 4 + 8 * ((r // 2) % 2), r % 2 + 2 * (l % 4) + 8 * (r // 4)
    else:
        raise ValueError(shape)
    return row, col


def ld_image(shape: str, n: int, tmem_word):
    """Registers every lane receives from ``tcgen05.ld.<shape>.x<n>`` given
    ``tmem_word(row, col)`` for the atom's rows/cols; returns (32, regs)."""
    regs = ld_regs_per_lane(shape, n)
    lanes = np.arange(32)[:, None]
    rr = np.arange(regs)[None, :]
    row, col = ld_owner(shape, lanes, rr)
    return tmem_word(row, col)


def split_owner(lane, reg, imm_lanes: int, imm_cols: int):
    """Split accesses ``16x32bx2`` ("tcgen05.ld / tcgen05.st" page, "Split
    accesses: 16x32bx2"): lane l owns (access l//16, row l%16, column r), and
    access 1 starts at the first address plus the immediate
    ``(imm_lanes << 16) + imm_cols`` -- lane 16 adds no sixteen-row shift of
    its own.  Returns the (lane, column) offset from the first address."""
    l = np.asarray(lane)
    r = np.asarray(reg)
    access = l // 16
    return l % 16 + access * imm_lanes + 0 * r, r + access * imm_cols + 0 * l


def split_load(num: int, imm_lanes: int, imm_cols: int, tmem_word):
    """Registers (32, num) that ``tcgen05.ld.16x32bx2.x<num>`` gives a warp,
    with ``tmem_word(lane, col)`` relative to the first address."""
    lanes = np.arange(32)[:, None]
    rr = np.arange(num)[None, :]
    return tmem_word(*split_owner(lanes, rr, imm_lanes, imm_cols))


def split_store(regs, imm_lanes: int, imm_cols: int, shape=(32, 32)):
    """Tensor-memory image (zero where nothing is written) that
    ``tcgen05.st.16x32bx2.x<num>`` of ``regs`` (32, num) leaves, relative to
    the first address.  Two registers landing on one cell is an error here:
    the page gives such a store no defined result."""
    regs = np.asarray(regs)
    lanes = np.arange(32)[:, None]
    rr = np.arange(regs.shape[1])[None, :]
    row, col = split_owner(lanes, rr, imm_lanes, imm_cols)
    if np.unique(row * 4096 + col).size != row.size:
        raise ValueError("the two accesses overlap")
    img = np.zeros(shape, dtype=regs.dtype)
    img[row, col] = regs
    return img


def layout_b_position(i, j):
    """Layout B ("tcgen05.ld / tcgen05.st" page, example): logical [i, j] of a
    (64, 128) tile sits at lane i + 64*(j//64), column j % 64."""
    i = np.asarray(i)
    j = np.asarray(j)
    return i + 64 * (j // 64), j % 64


def ws64_position(i, j, N: int):
    """Where a weight-stationary M = 64 MMA leaves accumulator element (i, j)
    of its 64 x N tile ("tcgen05.mma" page: "M64 .ws uses Layout E", and with
    A in TMEM "A ends in (2,64,K)"; "splitting an M64 N128 operation into two
    N64 issues changes each instruction's bank boundary from 64 to 32
    columns").  READING: the N columns split into two banks at N/2; bank
    b = j // (N/2) occupies lanes 64b .. 64b+63, so (i, j) sits at lane
    i + 64*(j // (N/2)), column j % (N/2) -- for N = 128 exactly the page's
    Layout B -- and a TMEM A operand holds one 64-row copy per bank, bank b
    in lanes 64b .. 64b+63, feeding that bank's columns.
    Returns (lane, column)."""
    i = np.asarray(i)
    j = np.asarray(j)
    half = N // 2
    return i + 64 * (j // half), j % half


# ---------------------------------------------------------------------------
# ldmatrix / stmatrix m8n8.b16 ("ldmatrix / stmatrix" page, "Address providers
# and result owners", "Transpose and stores").
# ---------------------------------------------------------------------------


def ldmatrix_address_provider(matrix: int, row: int) -> int:
    """Lane 8*matrix + row provides the shared address of that row."""
    return 8 * matrix + row


def ldmatrix_owner(matrix: int, row: int, word: int):
    """Register word (matrix, row, word) belongs to lane 4*row + word, in that
    lane's ``matrix``-th destination register."""
    return 4 * row + word, matrix


def ldmatrix_load(shared_rows, count: int, trans: bool = False):
    """Simulate ``ldmatrix.m8n8.x<count>[.trans].b16``.

    ``shared_rows[matrix][row]`` is the list of four b32 words (each two
    16-bit halves, low half first) of that 16-byte row, as supplied by the
    address-providing lane.  Returns regs[lane][matrix] as b32 ints.
    With .trans, register element (row, 2*word+half) comes from shared element
    (2*word+half, row) of the same 8x8 matrix of 16-bit values.
    """
    regs = [[None] * count for _ in range(32)]
    for m in range(count):
        halves = [[(shared_rows[m][r][c // 2] >> (16 * (c % 2))) & 0xFFFF for c in range(8)]
                  for r in range(8)]
        for row in range(8):
            for word in range(4):
                lane, reg = ldmatrix_owner(m, row, word)
                if trans:
                    lo = halves[2 * word][row]
                    hi = halves[2 * word + 1][row]
                else:
                    lo = halves[row][2 * word]
                    hi = halves[row][2 * word + 1]
                regs[lane][reg] = lo | (hi << 16)
    return regs


def stmatrix_store(regs, count: int, trans: bool = False):
    """Simulate ``stmatrix.m8n8.x<count>[.trans].b16`` ("Transpose and
    stores": the register image of the load is the store's input, each
    provider's row address its output).  ``regs[lane][matrix]`` are b32 ints;
    returns rows[matrix][row] = the four b32 words written to the 16-byte row
    whose address lane 8*matrix + row provides.  Register word
    (matrix, row, word) is lane 4*row + word's ``matrix``-th register; with
    .trans, shared element (r, c) of a matrix receives register element
    (c, r) of 16-bit values."""

    def reg_half(m, row, c):
        return (regs[4 * row + c // 2][m] >> (16 * (c % 2))) & 0xFFFF

    rows = []
    for m in range(count):
        mat = []
        for r in range(8):
            words = []
            for w in range(4):
                if trans:
                    lo, hi = reg_half(m, 2 * w, r), reg_half(m, 2 * w + 1, r)
                else:
                    lo, hi = reg_half(m, r, 2 * w), reg_half(m, r, 2 * w + 1)
                words.append(lo | (hi << 16))
            mat.append(words)
        rows.append(mat)
    return rows


# ---------------------------------------------------------------------------
# Block-scale factors in TMEM ("tcgen05.mma" page, "Weight-stationary and block
# scaling"; "tcgen05.cp" page, shape table).
# ---------------------------------------------------------------------------


def sf_tmem_position(r, sf):
    """Scale row r uses lane r%32 and byte-column 4*(r//32)+sf, with four
    replicas 32 lanes apart.  Returns (lanes[4], b32 column, byte in column)."""
    r = np.asarray(r)
    bytecol = 4 * (r // 32) + np.asarray(sf)
    lanes = np.stack([r % 32 + 32 * q for q in range(4)])
    return lanes, bytecol // 4, bytecol % 4


def cp_32x128b_warpx4_position(row, byte):
    """tcgen05.cp .32x128b.warpx4: a (32, 4)-word source image; source row i
    goes to 32 consecutive lanes (i) replicated four times 32 lanes apart;
    columns are consecutive b32 cells, so byte b of the 16-byte row lands in
    column b//4, byte b%4."""
    row = np.asarray(row)
    byte = np.asarray(byte)
    lanes = np.stack([row + 32 * q for q in range(4)])
    return lanes, byte // 4, byte % 4


def sf_chunk_offset(r, kb):
    """Byte offset, inside one 512-byte scale chunk (128 rows x 4 K blocks),
    at which the scale of row r and K block kb must sit so that one
    .32x128b.warpx4 copy puts it where the MMA reads it: 16*(r%32) +
    4*(r//32) + kb (source row r%32, byte 4*(r//32)+kb)."""
    r = np.asarray(r)
    return 16 * (r % 32) + 4 * (r // 32) + np.asarray(kb)


def sf_prepare(sf: np.ndarray, rows: int, kblocks: int, tile_rows: int) -> np.ndarray:
    """Rearrange plain row-major e8m0 scales ``sf[rows][kblocks]`` into the
    cp-ready image the kernels stream: for every K step of 4 scale blocks
    (128 K elements) and every tile of ``tile_rows`` rows, ceil(tile_rows/128)
    consecutive 512-byte chunks laid out by :func:`sf_chunk_offset`.
    Missing rows/blocks (ragged tails) hold 127 (a scale of 1.0; the matching
    operand values are zero-filled, so the value does not matter).
    Image order: [kstep][tile][chunk][512]."""
    ksteps = -(-kblocks // 4)
    tiles = -(-rows // tile_rows)
    chunks = -(-tile_rows // 128)
    out = np.full((ksteps, tiles, chunks, 512), 127, dtype=np.uint8)
    for t in range(tiles):
        for c in range(chunks):
            for rl in range(128):
                r = t * tile_rows + c * 128 + rl
                if rl + c * 128 >= tile_rows or r >= rows:
                    continue
                for ks in range(ksteps):
                    for kb in range(4):
                        kk = ks * 4 + kb
                        if kk < kblocks:
                            out[ks, t, c, int(sf_chunk_offset(rl, kb))] = sf[r, kk]
    return out
