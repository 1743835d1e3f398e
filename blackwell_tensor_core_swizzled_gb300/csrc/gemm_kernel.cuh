// Persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
//   D[m,n] = sum_k A[m,k] B[k,n]       (kind::f16, kind::tf32)
//   D[m,n] = sum_k (SFA.A)[m,k] (SFB.B)[k,n]   (kind::mxf8f6f4 / mxf4 / mxf4nvf4
//                                              .block_scale)
//
// Structure (one CTA per SM, or one CTA pair per two SMs for cta_group::2).
// The issuing roles run their loops on the whole warp in uniform control flow
// (one vote per barrier wait, warp-uniform operands) and one elected lane
// issues:
//   warp 0      TMA producer: 128B-swizzled A/B tiles (and scale images) into
//               a STAGES-deep ring, full[s] barriers counting bytes;
//   warp 1      MMA issuer (pair leader only): for each ring stage the scale
//               copies when it stages them (tcgen05.cp .32x128b.warpx4, the
//               default for block scaling), KSTEPS tcgen05.mma issues, then
//               tcgen05.commit -> empty[s]; at the end of a tile a commit ->
//               acc_full[b];
//   warp 2      TMEM allocation / deallocation (512 columns);
//   warp 3      barrier initialisation; with block scaling and
//               GemmParams::sf_mode SF_BY_CP a separate copy warp:
//               tcgen05.cp + commit -> sf_ready[slot];
//   warps 4..7  epilogue: tcgen05.ld .32x32b from accumulator b (warp w
//               reads lanes 32*(w%4)..+31), convert, store to global
//               (through a shared staging tile and a TMA tile store when
//               the output's alignment allows), then arrive acc_empty[b];
//   warps 8..11 (block scaling) with SF_BY_WARPS (8- and 6-bit formats
//               only): scale staging, each warp
//               writes its TMEM lane quadrant of the stage's scale slot with
//               tcgen05.st and arrives sf_ready[slot]; otherwise they join
//               the epilogue (the two warps of a lane quadrant drain
//               alternate 32-column chunks).
// With two accumulators the epilogue of one tile overlaps the main loop of the
// next.  With one (a 256-column block-scaled tile leaves no TMEM for a second)
// an eight-warp epilogue with 16-bit output reads the whole accumulator into
// registers, releases it, and only then converts and stores, so the next
// tile's MMAs wait for the TMEM reads alone.
//
// The MMA issue follows the "tcgen05.mma" page: one elected thread issues the
// K repeats as separate instructions with accumulation disabled only on the
// very first, and one commit covers the sequence; the epilogue follows the
// "tcgen05.ld / tcgen05.st" page's completion rules (commit, mbarrier wait,
// tcgen05.fence::after_thread_sync, ld, wait::ld).  Block-scale placement in
// TMEM is the page's "lane r%32, byte-column 4*(r//32)+sf, four replicas",
// produced by tcgen05.cp .32x128b.warpx4 ("tcgen05.cp" page, shape table).
//
// The kernel is launched as a programmatic dependent of the previous kernel on
// its stream (griddepcontrol.wait before any global access or TMEM allocation).
//
// Every mbarrier wait is bounded (GemmParams::timeout_ns); a wait that runs
// out records an error word, raises a CTA-local abort flag and the kernel
// drains its in-flight copies / MMAs (again bounded), frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "desc.cuh"
#include "ptx.cuh"

namespace tcg {

// KIND_MXF8: kind::mxf8f6f4 block-scaled (E4M3 / E5M2 / FP6 / padded FP4);
// KIND_MXF4 / KIND_NVF4: packed FP4, kind::mxf4 with two e8m0 scales per MMA
// row, kind::mxf4nvf4 with four unsigned E4M3 scales per MMA row.
enum Kind : int { KIND_F16 = 0, KIND_TF32 = 1, KIND_MXF8 = 2, KIND_MXF4 = 3, KIND_NVF4 = 4 };
enum OutType : int { OUT_F32 = 0, OUT_F16 = 1, OUT_BF16 = 2 };
enum SfMode : int { SF_BY_WARPS = 0, SF_BY_MMA = 1, SF_BY_CP = 2 };

// Error word layout: bits [0,8) status (1 = wait timeout), [8,16) site,
// [16,48) block index.
enum ErrSite : uint32_t {
  SITE_PROD_EMPTY = 1,
  SITE_MMA_FULL = 2,
  SITE_MMA_ACC_EMPTY = 3,
  SITE_EPI_ACC_FULL = 4,
  SITE_DRAIN = 5,
  SITE_PROBE = 6
};

struct GemmParams {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b;
  CUtensorMap tmap_sfa;
  CUtensorMap tmap_sfb;
  CUtensorMap tmap_d;  // D in 32-row x 64-byte boxes, 64-byte swizzle (used when d_tma)
  CUtensorMap tmap_w;  // fp32 partial-tile slots [slots][w_rows][BN] in 16 x 32 x 1 boxes, 64-byte swizzle
  int M, N, K;
  int num_m_tiles;   // tiles of 128*CG rows
  int num_n_tiles;   // tiles of BN columns
  int num_k_blocks;  // ring stages per tile (128 bytes of K each)
  // split-K: every output tile is computed by `split` units over consecutive
  // K ranges; num_units = num_tiles * split.  A unit that computes part of a
  // tile stores its fp32 partial into its own slot of the workspace `w`
  // ([slot * CG + rank][w_rows][BN], TMA stores through tmap_w in 16 x 32
  // boxes); splitk_reduce_kernel then sums each tile's slots into D.
  int split;
  int num_units;
  // stream-K: cluster c takes the global (tile, k block) iterations
  // [c*T/G, (c+1)*T/G), T = num_tiles * num_k_blocks, G = clusters, cut at
  // tile boundaries; a tile whose K blocks lie in one cluster is stored
  // directly, the others meet in the workspace like split-K units
  int stream_k;
  float* w;
  int w_rows;  // rows per slot: min(128, M)
  int bn;      // tile columns (BN of the kernel variant)
  int num_tiles;
  int raster_group;
  int a_mn_major, b_mn_major;
  int a_boxes, b_boxes;  // TMA boxes per stage (1 for K-major)
  int a_box_mn, b_box_mn;  // M/N extent of one MN-major box
  uint32_t a_box_bytes, b_box_bytes;
  // A and B bytes one stage brings in (both CTAs of a pair): the full tiles,
  // except that a single-CTA K-major A with M < 128 loads only round_up(M, 8)
  // rows (the rest of the smem tile is stale and feeds only rows >= M), and
  // that packed 6- / 4-bit elements count only their data bytes (TMA leaves
  // the padding of each 16-byte block unwritten)
  uint32_t ab_tx_bytes;
  uint64_t a_desc_hi, b_desc_hi;
  uint32_t a_kstep, b_kstep;  // descriptor start advance (bytes) per MMA K step
  uint32_t idesc;
  int sf_a_tiles;  // 128-row SFA tiles per K step in the scale image
  void* D;
  int64_t ldd;
  int d_type;
  int acc_f16;
  int d_vec_ok;
  // output stored by TMA from per-warp 32-row x 64-byte shared staging tiles
  // (32 columns of a 16-bit output, 16 of an fp32 one per tile)
  int d_tma;
  // the kernel computes the transposed product: its (row r, column c) is
  // D[c * ldd + r] (f32 accumulation, 32-column variant only; set by the host
  // for few-row problems whose operands it swapped)
  int d_trans;
  // 16-bit outputs through the staging tiles, fp32 accumulation: drain with
  // tcgen05.ld .16x256b (fragments) and write the staging tile with stmatrix
  // instead of .32x32b rows and st.shared.v4
  int epi_frag;
  unsigned long long* err;
  uint64_t timeout_ns;
  // block scaling, where the scales are staged into TMEM:
  //   SF_BY_WARPS  the four scale warps, tcgen05.st (scales complete on each
  //                CTA's own sf_loaded[s]);
  //   SF_BY_MMA    the MMA warp, tcgen05.cp before its MMAs;
  //   SF_BY_CP     a separate copy warp (warp 3), tcgen05.cp + commit to
  //                sf_ready[slot].
  // With tcgen05.cp (a pair copies both CTAs' smem) the scale images complete
  // on the pair leader's full[s] barrier together with A and B.
  int sf_mode;
  // optional phase trace (null: off): per CTA, TRACE_SLOTS globaltimer
  // stamps (see TraceSlot) and the number of units it processed
  unsigned long long* trace;
  int trace_ctas;
};

enum TraceSlot : int {
  TRACE_ENTRY = 0,        // kernel entry
  TRACE_SETUP = 1,        // barriers and TMEM ready
  TRACE_PRODUCER = 2,     // producer starts its first unit
  TRACE_FIRST_UNIT = 3,   // MMA warp has issued its first unit (pair leader / single CTA)
  TRACE_LAST_COMMIT = 4,  // last tile's accumulator committed (MMA warp)
  TRACE_EPI_DONE = 5,     // epilogue stores drained (warp 4)
  TRACE_EXIT = 6,         // TMEM released, CTA about to exit
  TRACE_UNITS = 7,        // units processed (MMA warp), not a time
  TRACE_CLK_ENTRY = 8,    // SM cycle counter next to TRACE_ENTRY
  TRACE_CLK_EXIT = 9,     // SM cycle counter next to TRACE_EXIT
  TRACE_SLOTS = 10
};

__device__ __forceinline__ void trace_stamp(const GemmParams& p, int slot) {
  if (p.trace && static_cast<int>(blockIdx.x) < p.trace_ctas)
    p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + slot] = globaltimer();
}

// A globaltimer stamp and the SM's cycle counter read back to back: the two
// pairs (entry, exit) give the CTA's average SM clock over the kernel.
__device__ __forceinline__ void trace_stamp_clock(const GemmParams& p, int slot, int clk_slot) {
  if (p.trace && static_cast<int>(blockIdx.x) < p.trace_ctas) {
    const uint64_t t = globaltimer();
    const uint64_t c = clock64();
    p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + slot] = t;
    p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + clk_slot] = c;
  }
}

// A_ROWS < 128 (single CTA, K-major A, M <= A_ROWS): only that many rows of
// A are staged per ring stage, so many more stages fit; the MMA still reads a
// 128-row operand, whose rows beyond A_ROWS are whatever follows in shared
// memory and only feed accumulator rows >= M, which are never stored.
//
// BN = 384 (block-scaled CTA pairs, K-major B): each K step issues two MMAs,
// N = 256 into accumulator columns 0..255 and N = 128 into 256..383.  A pair
// MMA of N columns reads N/2 B rows from each CTA at the same shared offset,
// the first CTA's giving columns [0, N/2); so CTA r stages tile columns
// 128r .. 128r+127 in its B rows 0..127 and 256+64r .. 256+64r+63 in rows
// 128..191 (three 64-row boxes), and accumulator column c is tile column c.
template <int CG, int BN, int ACC, int STAGES, int KIND, int A_ROWS = 128>
struct GemmCfg {
  static constexpr bool SCALED = KIND >= KIND_MXF8;  // block-scaled kinds
  static constexpr bool WIDE = BN > 256;             // two MMAs per K step
  static constexpr int BM = 128;            // accumulator rows per CTA
  static constexpr int BN_LOCAL = BN / CG;  // B rows staged per CTA
  static constexpr int A_BYTES = A_ROWS * 128;
  static constexpr int B_BYTES = BN_LOCAL * 128;
  static constexpr int SFB_CHUNKS = (BN + 127) / 128;
  // 512-byte scale chunks (128 rows x 4 scale bytes) per 128 rows per stage:
  // a stage holds 4 (MX 8/6-bit), 8 (MXFP4) or 16 (NVFP4) scales per row
  static constexpr int SF_KCH = KIND == KIND_MXF4 ? 2 : KIND == KIND_NVF4 ? 4 : 1;
  static constexpr int SFA_BYTES = SCALED ? 512 * SF_KCH : 0;
  static constexpr int SFB_BYTES = SCALED ? 512 * SFB_CHUNKS * SF_KCH : 0;
  static constexpr int LOAD_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  static constexpr int STAGE_BYTES = (LOAD_BYTES + 1023) / 1024 * 1024;
  // scale-image bytes of one stage (counted on the pair leader's full
  // barrier for both CTAs, or on each CTA's sf_loaded barrier)
  static constexpr int SF_TX_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int MMA_M = 128 * CG;
  static constexpr int MMA_K = KIND == KIND_F16 ? 16 : KIND == KIND_TF32 ? 8 : KIND == KIND_MXF8 ? 32 : 64;
  // K elements per stage: one 128-byte row (packed FP4: two per byte)
  static constexpr int BK = KIND == KIND_F16 ? 64 : KIND == KIND_TF32 ? 32 : KIND == KIND_MXF8 ? 128 : 256;
  static constexpr int KSTEPS = BK / MMA_K;    // MMA issues per stage
  // K extent of a stage in the operand maps' units: packed FP4 is mapped as
  // bytes, every other type in elements
  static constexpr int MAP_K = (KIND == KIND_MXF4 || KIND == KIND_NVF4) ? 128 : BK;
  // scale columns MMA issue j reads (relative to its slot): the chunk group of
  // its K, then the scale id (the byte within the column)
  static constexpr int SF_GROUP_MMAS = KSTEPS / SF_KCH;  // issues per 4-byte scale group
  __host__ __device__ static constexpr int sfa_col(int j) { return 4 * (j / SF_GROUP_MMAS); }
  __host__ __device__ static constexpr int sfb_col(int j) { return 4 * SF_KCH + 4 * SFB_CHUNKS * (j / SF_GROUP_MMAS); }
  __host__ __device__ static constexpr uint32_t sf_id(int j) {
    return static_cast<uint32_t>((j % SF_GROUP_MMAS) * (4 / SF_GROUP_MMAS));
  }
  static constexpr int SF_COL0 = ACC * BN;     // scale-factor slots follow the accumulators
  static constexpr int TMEM_COLS = 512;
  // a scale slot: SFA 4 columns per chunk group, then SFB 4 per 128 rows per
  // group (128-bit aligned column origins, as tcgen05.cp requires)
  static constexpr int SF_SLOT_COLS = 4 * SF_KCH * (1 + SFB_CHUNKS);
  // Scale slots rotate over the free TMEM columns; before a slot is
  // rewritten the MMA thread waits for the stage that last used it to retire.
  // With as many slots as ring stages the wait is implied: full[s] of
  // iteration it completes only after the producer saw empty[s] of it - STAGES,
  // i.e. after the MMAs that last read slot it % STAGES retired.
  static constexpr int SF_SLOTS_FREE = (TMEM_COLS - ACC * BN) / SF_SLOT_COLS;
  static constexpr int SF_SLOTS = !SCALED ? 1 : SF_SLOTS_FREE < STAGES ? SF_SLOTS_FREE : STAGES;
  static constexpr bool SF_SLOT_WAIT = SF_SLOTS < STAGES;
  // epilogue staging for TMA stores: per epilogue warp EPI_BUFS tiles of
  // 32 rows x 64 bytes (32 16-bit columns), 64-byte swizzled
  static constexpr int EPI_WARPS_MAX = SCALED ? 8 : 4;
  static constexpr int EPI_BUFS = SCALED ? 1 : 2;
  static constexpr int EPI_TILE_BYTES = 32 * 64;
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS_MAX * EPI_BUFS * EPI_TILE_BYTES;
  // full[S], empty[S], acc_full[ACC], acc_empty[ACC], drain, and for block
  // scaling sf_loaded[S] (scale bytes in smem) and sf_ready[SF_SLOTS] (scales
  // written to TMEM by the scale warps)
  static constexpr int NUM_BARS = 2 * STAGES + 2 * ACC + 1 + (SCALED ? STAGES + SF_SLOTS : 0);
  static constexpr int SMEM_BYTES = 1024 + BAR_OFF + NUM_BARS * 8 + 16;
  // warps 0..7 as described above; block scaling adds warps 8..11, one per
  // TMEM lane quadrant, which stage the scale factors into TMEM
  static constexpr int THREADS = SCALED ? 384 : 256;
  // epilogue warps: 4..7, plus 8..11 when block scales are staged by tcgen05.cp
  __host__ __device__ static constexpr int epi_warps(int sf_mode) {
    return SCALED && sf_mode != SF_BY_WARPS ? 8 : 4;
  }
  static_assert(BN % 32 == 0 && BN >= 32 && (BN <= 256 || (BN == 384 && CG == 2 && SCALED && ACC == 1)),
                "epilogue drains 32-column chunks; MMA N <= 256 except the two-MMA pair tile");
  static_assert(BN % (16 * CG) == 0, "MMA N constraint / per-CTA B split");
  static_assert(ACC * BN + (SCALED ? SF_SLOTS * SF_SLOT_COLS : 0) <= TMEM_COLS, "TMEM budget");
  static_assert(!SCALED || (SF_SLOTS >= 1 && SF_SLOTS <= STAGES), "scale slots");
  static_assert(KSTEPS % SF_KCH == 0, "scale groups split the stage's MMAs evenly");
  static_assert(SMEM_BYTES <= 232448, "dynamic shared memory");
  static_assert(A_ROWS % 8 == 0 && A_ROWS <= 128 && (A_ROWS == 128 || CG == 1), "staged A rows");
  // the MMA's 128-row read of the last stage's A tile stays inside the
  // allocation (it runs into that stage's B tile and the epilogue staging)
  static_assert(BAR_OFF - (STAGES - 1) * STAGE_BYTES >= BM * 128, "A over-read in bounds");
};

struct WaitCtx {
  uint64_t timeout_ns;
  unsigned long long* err;
  volatile uint32_t* abort_flag;
};

__device__ __forceinline__ unsigned long long make_err(uint32_t status, uint32_t site) {
  return static_cast<unsigned long long>(status) | (static_cast<unsigned long long>(site) << 8) |
         (static_cast<unsigned long long>(blockIdx.x) << 16);
}

// Bounded parity wait by the calling thread.  Returns false on timeout (error
// recorded, abort raised) or when another role already aborted.
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, WaitCtx w, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (globaltimer() - t0 > w.timeout_ns) {
      *w.abort_flag = 1u;
      if (w.err) atomicCAS(w.err, 0ull, make_err(1u, site));
      return false;
    }
  }
}

// Every lane waits (each gets its own acquire), the outcome is made uniform
// across the warp.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, WaitCtx w, uint32_t site) {
  const bool ok = wait_bounded(bar, parity, w, site);
  return __all_sync(0xffffffffu, ok);
}

// Warp-uniform wait for the single-issuer roles: one vote when the phase has
// already completed (the common case), else every lane's bounded wait.
__device__ __forceinline__ bool wait_uniform(uint32_t bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_try_wait(bar, parity)) || warp_wait(bar, parity, w, site);
}

// CTA-wide barrier 0 without the .aligned restriction: the threads of a warp
// may arrive at different times (the single-thread roles finish after the
// rest of their warp).
__device__ __forceinline__ void cta_barrier_unaligned() { asm volatile("barrier.sync 0;" ::: "memory"); }

__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mt, int& nt) {
  const int G = p.raster_group;
  const int per_group = G * p.num_n_tiles;
  const int g = t / per_group;
  const int first_m = g * G;
  const int gs = min(p.num_m_tiles - first_m, G);
  const int r = t - g * per_group;
  mt = first_m + r % gs;
  nt = r / gs;
}

// The units (one tile's K blocks [kb0, kb1)) a cluster processes, in order:
// whole tiles cluster_id, +G, ... (split == 1); `split` consecutive K ranges
// per tile, unit u -> tile u / split (split > 1); or the cluster's stream-K
// range of the global iteration space, cut at tile boundaries.
struct UnitCursor {
  int64_t i, i1;   // stream-K position and end
  int u;           // strided unit index
  int first_tile;  // stream-K: the tile the cluster's range starts in
  int tile, kb0, kb1;
  bool valid;
};

__device__ __forceinline__ void cursor_load(UnitCursor& c, const GemmParams& p) {
  if (p.stream_k) {
    c.valid = c.i < c.i1;
    if (!c.valid) return;
    c.tile = static_cast<int>(c.i / p.num_k_blocks);
    const int64_t t0 = static_cast<int64_t>(c.tile) * p.num_k_blocks;
    c.kb0 = static_cast<int>(c.i - t0);
    c.kb1 = static_cast<int>(min(static_cast<int64_t>(p.num_k_blocks), c.i1 - t0));
  } else {
    c.valid = c.u < p.num_units;
    if (!c.valid) return;
    if (p.split == 1) {  // whole tiles: no divisions
      c.tile = c.u;
      c.kb0 = 0;
      c.kb1 = p.num_k_blocks;
      return;
    }
    c.tile = c.u / p.split;
    const int ks = c.u - c.tile * p.split;
    c.kb0 = static_cast<int>(static_cast<int64_t>(ks) * p.num_k_blocks / p.split);
    c.kb1 = static_cast<int>(static_cast<int64_t>(ks + 1) * p.num_k_blocks / p.split);
  }
}

__device__ __forceinline__ UnitCursor cursor_begin(int cluster_id, int num_clusters, const GemmParams& p) {
  UnitCursor c;
  c.u = cluster_id;
  c.i = c.i1 = 0;
  c.first_tile = 0;
  if (p.stream_k) {  // 64-bit divisions only where the stream-K range needs them
    const int64_t T = static_cast<int64_t>(p.num_tiles) * p.num_k_blocks;
    c.i = cluster_id * T / num_clusters;
    c.i1 = (cluster_id + 1) * T / num_clusters;
    c.first_tile = static_cast<int>(c.i / p.num_k_blocks);
  }
  cursor_load(c, p);
  return c;
}

__device__ __forceinline__ void cursor_next(UnitCursor& c, int num_clusters, const GemmParams& p) {
  if (p.stream_k)
    c.i = static_cast<int64_t>(c.tile + 1) * p.num_k_blocks;
  else
    c.u += num_clusters;
  cursor_load(c, p);
}

// Workspace slot of a partial unit: under stream-K a cluster has at most one
// partial unit at each end of its range (head: its first tile, tail: any
// later tile); under split-K the unit index.
__device__ __forceinline__ int unit_slot(const UnitCursor& c, int cluster_id, const GemmParams& p) {
  return p.stream_k ? 2 * cluster_id + (c.tile != c.first_tile ? 1 : 0) : c.u;
}

// Ring iterations (k blocks) of all units a cluster processes.
__device__ __forceinline__ uint32_t cluster_iterations(int cluster_id, int num_clusters, const GemmParams& p) {
  uint32_t n = 0;
  for (UnitCursor c = cursor_begin(cluster_id, num_clusters, p); c.valid; cursor_next(c, num_clusters, p))
    n += static_cast<uint32_t>(c.kb1 - c.kb0);
  return n;
}

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16(uint32_t lo, uint32_t hi) {
  __half2 v = __floats2half2_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

// Store 32 consecutive output columns of one row from 16 packed 16-bit pairs.
__device__ __forceinline__ void store_row16(const GemmParams& p, int row, int col0, const uint32_t (&h)[16]) {
  const int ncols = min(32, p.N - col0);
  uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + static_cast<int64_t>(row) * p.ldd + col0;
  if (ncols == 32 && p.d_vec_ok) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d4[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) dst[i] = static_cast<uint16_t>((h[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
  }
}

// Store 32 consecutive fp32 accumulator columns of one row, converted.
__device__ __forceinline__ void store_row32(const GemmParams& p, int row, int col0, const uint32_t (&r)[32]) {
  if (p.d_type == OUT_F32) {
    const int ncols = min(32, p.N - col0);
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.D) + static_cast<int64_t>(row) * p.ldd + col0;
    if (ncols == 32 && p.d_vec_ok) {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int i = 0; i < 8; ++i) d4[i] = make_uint4(r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < ncols) dst[i] = r[i];
    }
  } else {
    uint32_t h[16];
    if (p.d_type == OUT_BF16) {
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = pack_bf16(r[2 * i], r[2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = pack_f16(r[2 * i], r[2 * i + 1]);
    }
    store_row16(p, row, col0, h);
  }
}

// Store 32 fp32 accumulator columns of one row of the transposed product:
// column col0 + i goes to D[(col0 + i) * ldd + row], converted.  The 32 lanes
// of a warp hold consecutive rows, so each column is one contiguous run.
__device__ __forceinline__ void store_col32(const GemmParams& p, int row, int col0, const uint32_t (&r)[32]) {
  const int ncols = min(32, p.N - col0);
  const int64_t base = static_cast<int64_t>(col0) * p.ldd + row;
  if (p.d_type == OUT_F32) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.D) + base;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < ncols) dst[static_cast<int64_t>(i) * p.ldd] = r[i];
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + base;
    const bool bf = p.d_type == OUT_BF16;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < ncols) {
        const float v = __uint_as_float(r[i]);
        dst[static_cast<int64_t>(i) * p.ldd] =
            bf ? __bfloat16_as_ushort(__float2bfloat16_rn(v)) : __half_as_ushort(__float2half_rn(v));
      }
    }
  }
}

template <int CG, int BN, int ACC, int STAGES, int KIND, int A_ROWS = 128>
__global__ void __launch_bounds__(KIND >= KIND_MXF8 ? 384 : 256, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<CG, BN, ACC, STAGES, KIND, A_ROWS>;
  if (threadIdx.x == 0) trace_stamp_clock(p, TRACE_ENTRY, TRACE_CLK_ENTRY);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::BAR_OFF;
  // barrier addresses
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + ACC + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 2 * ACC);
  auto sfl_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + 2 * ACC + 1 + s); };
  auto sfr_bar = [&](int slot) { return bar0 + 8u * (3 * STAGES + 2 * ACC + 1 + slot); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::BAR_OFF + 8 * C::NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = (CG == 2) ? cluster_ctarank() : 0u;
  const int cluster_id = blockIdx.x / CG;
  const int num_clusters = gridDim.x / CG;
  const WaitCtx wctx{p.timeout_ns, p.err, abort_flag};

  // Prologue.  The roles' first unit (parameter reads, integer divisions)
  // and the producer's first tile coordinates are computed while warp 3
  // initialises the barriers and warp 2 allocates TMEM, so the first TMA
  // copies leave right after the setup barrier.
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b);
    if constexpr (C::SCALED) {
      prefetch_tmap(&p.tmap_sfa);
      prefetch_tmap(&p.tmap_sfb);
    }
  }
  UnitCursor uc_first{};
  int mt_first = 0, nt_first = 0;
  if (warp != 2 && warp != 3) {
    uc_first = cursor_begin(cluster_id, num_clusters, p);
    if (warp == 0 && uc_first.valid) tile_coords(uc_first.tile, p, mt_first, nt_first);
  }
  if (threadIdx.x == 96) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < ACC; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), C::epi_warps(p.sf_mode) * CG);
    }
    mbar_init(drain_bar, 1);
    if constexpr (C::SCALED) {
      for (int s = 0; s < STAGES; ++s) mbar_init(sfl_bar(s), 1);
      // sf_ready: one arrival per scale warp of each CTA, or one commit
      for (int k = 0; k < C::SF_SLOTS; ++k) mbar_init(sfr_bar(k), p.sf_mode == SF_BY_WARPS ? 4 * CG : 1);
    }
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  // The kernel is launched as a programmatic dependent of the previous kernel
  // on the stream: the prologue above overlaps that kernel's tail, and
  // griddepcontrol.wait returns once it has completed and its memory is
  // visible.  Every global access, and the TMEM allocation (a predecessor on
  // this SM may still hold columns), comes after the wait.
  griddep_wait();
  if (warp == 2) {
    tmem_alloc<CG>(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (threadIdx.x == 0) trace_stamp(p, TRACE_SETUP);
  // the next kernel on the stream may launch now; it waits for this grid's
  // completion before it touches memory
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop in uniform control flow (tile coordinates,
    // addresses and the tensor-map operands stay warp-uniform) and waits with
    // one vote; one elected lane issues the copies.  A lane-0-only loop
    // measured markedly slower.
    {
      uint32_t it = 0, s = 0, ph = 0;  // ring iteration, stage, phase of stage s
      bool ok = true;
      bool first_unit = true;
      if (lane == 0) trace_stamp(p, TRACE_PRODUCER);
      for (UnitCursor uc = uc_first; uc.valid && ok; cursor_next(uc, num_clusters, p)) {
        int mt = mt_first, nt = nt_first;
        if (!first_unit) tile_coords(uc.tile, p, mt, nt);
        first_unit = false;
        const int kb0 = uc.kb0, kb1 = uc.kb1;
        const int m0 = mt * C::MMA_M + static_cast<int>(rank) * C::BM;
        const int n0 = nt * BN + static_cast<int>(rank) * C::BN_LOCAL;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait_uniform(empty_bar(s), ph ^ 1u, wctx, SITE_PROD_EMPTY)) {
            ok = false;
            break;
          }
          if (elect_one()) {
          const uint32_t fb = (CG == 2) ? mapa_shared(full_bar(s), 0) : full_bar(s);
          const bool sf_on_full = C::SCALED && p.sf_mode != SF_BY_WARPS;
          if (rank == 0)
            mbar_arrive_expect_tx(full_bar(s), p.ab_tx_bytes + (sf_on_full ? C::SF_TX_BYTES * CG : 0));
          const uint32_t sa = sbase + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          const int k0 = kb * C::MAP_K;
          if (!p.a_mn_major) {
            tma_load<CG>(sa, &p.tmap_a, k0, m0, fb);
          } else {
            for (int i = 0; i < p.a_boxes; ++i) tma_load<CG>(sa + i * p.a_box_bytes, &p.tmap_a, m0 + i * p.a_box_mn, k0, fb);
          }
          if constexpr (C::WIDE) {
            // 64-row boxes: tile columns 128r + [0, 128) and 256 + 64r + [0, 64)
            const int nb = nt * BN;
            tma_load<CG>(sb, &p.tmap_b, k0, nb + 128 * static_cast<int>(rank), fb);
            tma_load<CG>(sb + 64 * 128, &p.tmap_b, k0, nb + 128 * static_cast<int>(rank) + 64, fb);
            tma_load<CG>(sb + 128 * 128, &p.tmap_b, k0, nb + 256 + 64 * static_cast<int>(rank), fb);
          } else if (!p.b_mn_major) {
            tma_load<CG>(sb, &p.tmap_b, k0, n0, fb);
          } else {
            for (int i = 0; i < p.b_boxes; ++i) tma_load<CG>(sb + i * p.b_box_bytes, &p.tmap_b, n0 + i * p.b_box_mn, k0, fb);
          }
          if constexpr (C::SCALED) {
            const uint32_t ssfa = sb + C::B_BYTES;
            const uint32_t ssfb = ssfa + C::SFA_BYTES;
            // a pair tile's second half may lie wholly beyond M: its A rows are
            // zero-filled, so any valid scale row will do.  The scale maps have
            // one 512-byte chunk per row; a stage's chunks are consecutive rows.
            const int sfa_tile = min(mt * CG + static_cast<int>(rank), p.sf_a_tiles - 1);
            const int ya = (kb * p.sf_a_tiles + sfa_tile) * C::SF_KCH;
            const int yb = (kb * p.num_n_tiles + nt) * C::SF_KCH * C::SFB_CHUNKS;
            if (sf_on_full) {
              // a tcgen05.cp of a pair reads both CTAs' smem: complete with A, B
              tma_load<CG>(ssfa, &p.tmap_sfa, 0, ya, fb);
              tma_load<CG>(ssfb, &p.tmap_sfb, 0, yb, fb);
            } else {
              // the scale warps of this CTA consume these: they complete on
              // this CTA's own sf_loaded[s]
              mbar_arrive_expect_tx(sfl_bar(s), C::SF_TX_BYTES);
              tma_load_2d(ssfa, &p.tmap_sfa, 0, ya, sfl_bar(s));
              tma_load_2d(ssfb, &p.tmap_sfb, 0, yb, sfl_bar(s));
            }
          }
          }
          __syncwarp();
          ++it;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && elect_one()) {
        // Drain: let the copies this CTA issued land before the CTA can exit.
        const uint32_t n_out = it < static_cast<uint32_t>(STAGES) ? it : static_cast<uint32_t>(STAGES);
        if (KIND == KIND_MXF8 && p.sf_mode == SF_BY_WARPS) {
          for (uint32_t j = it - n_out; j < it; ++j) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(sfl_bar(j % STAGES), (j / STAGES) & 1u) && globaltimer() - t0 < 20000000ull) {
            }
          }
        }
        if (CG == 1 || rank == 0) {
          for (uint32_t j = it - n_out; j < it; ++j) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full_bar(j % STAGES), (j / STAGES) & 1u) && globaltimer() - t0 < 20000000ull) {
            }
          }
        } else {
          const uint64_t t0 = globaltimer();
          while (globaltimer() - t0 < 2000000ull) {
          }
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The pair leader's warp 1.  The tensor pipe queues little ahead of the
    // MMAs it executes, so the per-stage path must be short: the warp runs
    // the loop in uniform control flow (descriptors are warp-uniform values:
    // the stage-0 descriptors plus precomputed stage / K-step increments),
    // waits with one vote, and one elected lane issues the MMAs and commits.
    // Issuing from a lane-0-only branch measured slower.  The loop is
    // compiled once per scale-staging mode, so the per-stage path carries no
    // runtime test of the mode (1.5 % at MXFP8 8192^3).
    auto mma_role = [&](auto sf_mode_tag) {
      constexpr int SFM = decltype(sf_mode_tag)::value;
      const uint64_t a_desc0 = sdesc(sbase, p.a_desc_hi);
      const uint64_t b_desc0 = sdesc(sbase + C::A_BYTES, p.b_desc_hi);
      const uint64_t a_step = p.a_kstep >> 4, b_step = p.b_kstep >> 4;  // 16-byte units
      uint32_t idesc_j[C::KSTEPS];
#pragma unroll
      for (int j = 0; j < C::KSTEPS; ++j)
        idesc_j[j] = C::SCALED ? (p.idesc | idesc_sf_ids(C::sf_id(j), C::sf_id(j))) : p.idesc;
      // block scales staged by other threads: wait for sf_ready[slot] too
      constexpr bool sf_wait = C::SCALED && SFM != SF_BY_MMA;
      constexpr bool sf_by_mma = C::SCALED && SFM == SF_BY_MMA;
      // the copy warp commits sf_ready[slot] only after it saw full[s] of the
      // same iteration, so that one wait covers both
      constexpr bool full_via_sfr = C::SCALED && SFM == SF_BY_CP;
      uint32_t it = 0, s = 0, ph = 0, tcount = 0;
      bool ok = true;
      for (UnitCursor uc = uc_first; uc.valid && ok; cursor_next(uc, num_clusters, p), ++tcount) {
        const int kb0 = uc.kb0, kb1 = uc.kb1;
        const int b = static_cast<int>(tcount % ACC);
        const uint32_t aph = (tcount / ACC) & 1u;
        if (!wait_uniform(acce_bar(b), aph ^ 1u, wctx, SITE_MMA_ACC_EMPTY)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          const uint32_t slot = it % C::SF_SLOTS;
          if (!full_via_sfr && !wait_uniform(full_bar(s), ph, wctx, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          if (sf_wait && !wait_uniform(sfr_bar(slot), (it / C::SF_SLOTS) & 1u, wctx, SITE_MMA_FULL)) {
            // the scale warps of both CTAs (tcgen05.st) or the copy warp
            // (tcgen05.cp + commit) fill this iteration's slot
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t st = (s * static_cast<uint32_t>(C::STAGE_BYTES)) >> 4;
          const uint64_t adesc = a_desc0 + st;
          const uint64_t bdesc = b_desc0 + st;
          const uint32_t sf_col = tmem_base + C::SF_COL0 + slot * C::SF_SLOT_COLS;
          if constexpr (sf_by_mma) {
            // this thread stages the scales with tcgen05.cp; they arrived
            // with full[s].  The slot's previous readers (the MMAs of
            // iteration it - SF_SLOTS) must have completed.
            if (C::SF_SLOT_WAIT && it >= static_cast<uint32_t>(C::SF_SLOTS)) {
              const uint32_t j = it - C::SF_SLOTS;
              if (!wait_uniform(empty_bar(j % STAGES), (j / STAGES) & 1u, wctx, SITE_MMA_FULL)) {
                ok = false;
                break;
              }
            }
            const uint32_t ssfa = sbase + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
            // 32 rows x 16 bytes, rows 16 bytes apart: (ldo 16, sdo 128, no swizzle)
            const uint64_t cp_hi = sdesc_hi(16, 128, SW_NONE);
            if (elect_one()) {
              // chunk group g (4 scales per row) of SFA to columns 4g; of SFB,
              // 128-row chunk c of group g to 4*SF_KCH + 4*(g*SFB_CHUNKS + c)
#pragma unroll
              for (int g = 0; g < C::SF_KCH; ++g)
                tc_cp_32x128b_warpx4<CG>(sf_col + 4 * g, sdesc(ssfa + 512 * g, cp_hi));
#pragma unroll
              for (int g = 0; g < C::SF_KCH; ++g)
#pragma unroll
                for (int c = 0; c < C::SFB_CHUNKS; ++c)
                  tc_cp_32x128b_warpx4<CG>(sf_col + 4 * C::SF_KCH + 4 * (g * C::SFB_CHUNKS + c),
                                           sdesc(ssfa + C::SFA_BYTES + 512 * (g * C::SFB_CHUNKS + c), cp_hi));
            }
          }
          if (elect_one()) {
#pragma unroll
          for (int j = 0; j < C::KSTEPS; ++j) {
            const uint64_t ad = adesc + j * a_step;
            const uint64_t bd = bdesc + j * b_step;
            const uint32_t acc = (kb != kb0 || j != 0) ? 1u : 0u;
            if constexpr (KIND == KIND_MXF8)
              mma_mxf8<CG>(d_tmem, ad, bd, idesc_j[j], sf_col + C::sfa_col(j), sf_col + C::sfb_col(j), acc);
            else if constexpr (KIND == KIND_MXF4)
              mma_mxf4<CG>(d_tmem, ad, bd, idesc_j[j], sf_col + C::sfa_col(j), sf_col + C::sfb_col(j), acc);
            else if constexpr (KIND == KIND_NVF4)
              mma_nvf4<CG>(d_tmem, ad, bd, idesc_j[j], sf_col + C::sfa_col(j), sf_col + C::sfb_col(j), acc);
            else if constexpr (KIND == KIND_F16)
              mma_f16<CG>(d_tmem, ad, bd, idesc_j[j], acc);
            else
              mma_tf32<CG>(d_tmem, ad, bd, idesc_j[j], acc);
            if constexpr (C::WIDE) {
              // BN = 384: the second issue, of the same kind (WIDE implies a
              // block-scaled kind), has N = 128 (p.idesc carries 256), reads B
              // rows 128.. (16 KiB on) and the third SFB chunk
              constexpr uint32_t N_FIELD = 0x3Fu << 17;
              constexpr uint32_t N128 = (128u >> 3) << 17;
              constexpr uint64_t B_HI_OFF = (128u * 128u) >> 4;
              const uint32_t id2 = (idesc_j[j] & ~N_FIELD) | N128;
              const uint32_t sfb2 = sf_col + C::sfb_col(j) + 8;
              if constexpr (KIND == KIND_MXF8)
                mma_mxf8<CG>(d_tmem + 256, ad, bd + B_HI_OFF, id2, sf_col + C::sfa_col(j), sfb2, acc);
              else if constexpr (KIND == KIND_MXF4)
                mma_mxf4<CG>(d_tmem + 256, ad, bd + B_HI_OFF, id2, sf_col + C::sfa_col(j), sfb2, acc);
              else
                mma_nvf4<CG>(d_tmem + 256, ad, bd + B_HI_OFF, id2, sf_col + C::sfa_col(j), sfb2, acc);
            }
          }
          tc_commit<CG>(empty_bar(s));
          }
          __syncwarp();
          ++it;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit<CG>(accf_bar(b));
        __syncwarp();
        if (tcount == 0 && lane == 0) trace_stamp(p, TRACE_FIRST_UNIT);
      }
      if (lane == 0) {
        trace_stamp(p, TRACE_LAST_COMMIT);
        if (p.trace && static_cast<int>(blockIdx.x) < p.trace_ctas)
          p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + TRACE_UNITS] = tcount;
      }
      if (!ok && elect_one()) {
        // Drain: wait (bounded) for every MMA / cp this thread issued.
        tc_commit<CG>(drain_bar);
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < 20000000ull) {
        }
      }
      __syncwarp();
    };
    if (CG == 1 || rank == 0) {
      if constexpr (KIND == KIND_MXF8) {
        if (p.sf_mode == SF_BY_MMA)
          mma_role(std::integral_constant<int, SF_BY_MMA>{});
        else if (p.sf_mode == SF_BY_CP)
          mma_role(std::integral_constant<int, SF_BY_CP>{});
        else
          mma_role(std::integral_constant<int, SF_BY_WARPS>{});
      } else if constexpr (C::SCALED) {
        // packed FP4: the MMA warp or a copy warp stages the scales
        if (p.sf_mode == SF_BY_CP)
          mma_role(std::integral_constant<int, SF_BY_CP>{});
        else
          mma_role(std::integral_constant<int, SF_BY_MMA>{});
      } else {
        mma_role(std::integral_constant<int, SF_BY_MMA>{});
      }
    }
  } else if (C::SCALED && warp == 3) {
    // ------------------------------------------------------------ cp thread
    // SF_BY_CP: the pair leader's warp 3 copies each stage's scales into its
    // TMEM slot with tcgen05.cp .32x128b.warpx4 (both CTAs of a pair) and
    // commits to sf_ready[slot]; the MMA warp's tensor-pipe stream then holds
    // only MMAs.  Uniform loop, one elected lane issues (as for the MMAs).
    if constexpr (C::SCALED) {
      if (p.sf_mode == SF_BY_CP && (CG == 1 || rank == 0)) {
        const uint32_t total_it = cluster_iterations(cluster_id, num_clusters, p);
        const uint64_t cp_hi = sdesc_hi(16, 128, SW_NONE);  // 32 rows x 16 B, rows 16 B apart
        uint32_t s = 0, ph = 0, issued = 0;
        for (uint32_t it = 0; it < total_it; ++it) {
          if (!wait_uniform(full_bar(s), ph, wctx, SITE_MMA_FULL)) break;
          if (C::SF_SLOT_WAIT && it >= static_cast<uint32_t>(C::SF_SLOTS)) {
            const uint32_t j = it - C::SF_SLOTS;  // the slot's previous readers
            if (!wait_uniform(empty_bar(j % STAGES), (j / STAGES) & 1u, wctx, SITE_MMA_FULL)) break;
          }
          tc_fence_after();
          const uint32_t ssfa = sbase + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
          const uint32_t col = tmem_base + C::SF_COL0 + (it % C::SF_SLOTS) * C::SF_SLOT_COLS;
          if (elect_one()) {
            // the slot layout the MMA path's copies produce: chunk group g of
            // SFA to columns 4g, 128-row chunk c of group g of SFB to
            // 4*SF_KCH + 4*(g*SFB_CHUNKS + c)
#pragma unroll
            for (int g = 0; g < C::SF_KCH; ++g)
              tc_cp_32x128b_warpx4<CG>(col + 4 * g, sdesc(ssfa + 512 * g, cp_hi));
#pragma unroll
            for (int g = 0; g < C::SF_KCH; ++g)
#pragma unroll
              for (int c = 0; c < C::SFB_CHUNKS; ++c)
                tc_cp_32x128b_warpx4<CG>(col + 4 * C::SF_KCH + 4 * (g * C::SFB_CHUNKS + c),
                                         sdesc(ssfa + C::SFA_BYTES + 512 * (g * C::SFB_CHUNKS + c), cp_hi));
            tc_commit<CG>(sfr_bar(it % C::SF_SLOTS));
          }
          __syncwarp();
          issued = it + 1;
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (issued > 0 && elect_one()) {
          // let the copies land before the CTA can exit: the last commit
          // tracks every copy this thread issued
          const uint32_t j = issued - 1;
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(sfr_bar(j % C::SF_SLOTS), (j / C::SF_SLOTS) & 1u) &&
                 globaltimer() - t0 < 20000000ull) {
          }
        }
      }
    }
  } else if (KIND == KIND_MXF8 && warp >= 8 && p.sf_mode == SF_BY_WARPS) {
    // ------------------------------------------------------------ scale warps
    // Warp 8+q writes TMEM lane quadrant q of every scale slot: source row l
    // of a 512-byte chunk (bytes [16l, 16l+16)) goes to lane 32q + l, four
    // columns, which is the placement one tcgen05.cp .32x128b.warpx4 of the
    // chunk produces (each quadrant is one of its replicas).
    if constexpr (KIND == KIND_MXF8) {
      if (p.sf_mode == SF_BY_WARPS) {
        const int q = warp & 3;
        const uint32_t total_it = cluster_iterations(cluster_id, num_clusters, p);
        uint32_t s = 0, ph = 0;
        for (uint32_t it = 0; it < total_it; ++it) {
          if (!warp_wait(sfl_bar(s), ph, wctx, SITE_MMA_FULL)) break;
          if (C::SF_SLOT_WAIT && it >= static_cast<uint32_t>(C::SF_SLOTS)) {
            // the slot's previous readers: the MMAs of iteration it - SF_SLOTS
            const uint32_t j = it - C::SF_SLOTS;
            if (!warp_wait(empty_bar(j % STAGES), (j / STAGES) & 1u, wctx, SITE_MMA_FULL)) break;
          }
          tc_fence_after();
          const uint4* sf = reinterpret_cast<const uint4*>(gbase + s * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES);
          const uint32_t slot = it % C::SF_SLOTS;
          const uint32_t col =
              tmem_base + (static_cast<uint32_t>(32 * q) << 16) + C::SF_COL0 + slot * C::SF_SLOT_COLS;
          tmem_st_32x32b_x4(col, sf[lane]);  // SFA: 4 columns
#pragma unroll
          for (int c = 0; c < C::SFB_CHUNKS; ++c) tmem_st_32x32b_x4(col + 4 + 4 * c, sf[32 * (1 + c) + lane]);  // SFB
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (CG == 2)
              mbar_arrive_cluster(mapa_shared(sfr_bar(slot), 0));
            else
              mbar_arrive(sfr_bar(slot));
          }
          if (++s == STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int nparts = C::epi_warps(p.sf_mode) / 4;
    const int part = (warp - 4) >> 2;        // this warp drains chunks part, part + nparts, ...
    // one accumulator, eight warps, 16-bit output: read everything, release, then store
    const bool early = ACC == 1 && nparts == 2 && (p.acc_f16 || p.d_type != OUT_F32);
    // transposed stores exist in the 32-column f16/bf16 variant only
    constexpr bool TRANS = BN == 32 && KIND == KIND_F16;
    // TMA-store staging: this warp's EPI_BUFS tiles of 32 rows x 64 bytes
    const uint32_t epi_base = sbase + C::EPI_OFF + static_cast<uint32_t>((warp - 4) * C::EPI_BUFS * C::EPI_TILE_BYTES);
    uint32_t epi_n = 0;
    // Store the warp's 32 x 32 block of 16-bit outputs (lane = row) at
    // (row0, col0): each row's four 16-byte chunks go to the staging tile in
    // the 64-byte swizzle (chunk j at j ^ ((row >> 1) & 3)), one lane issues
    // the tile store; the tensor map clips rows >= M and columns >= N.
    // to_slot: (col0, row0, z) address the workspace slot map instead of D
    // frag: h holds fragments (frag_load16's order) written with stmatrix,
    // each matrix an 8-row x 16-byte block of the same swizzled tile.
    auto stage_tile = [&](int row0, int col0, const uint32_t(&h)[16], bool to_slot, int z, bool frag = false) {
      const uint32_t buf = epi_base + (epi_n % C::EPI_BUFS) * C::EPI_TILE_BYTES;
      if (epi_n >= static_cast<uint32_t>(C::EPI_BUFS)) {
        if (lane == 0) bulk_wait_group_read<C::EPI_BUFS - 1>();  // the buffer's last store has read it
        __syncwarp();
      }
      if (frag) {
        // lane 8m + i addresses row i of matrix m (16-byte chunk m of its row)
        const uint32_t m = static_cast<uint32_t>(lane) >> 3, i = static_cast<uint32_t>(lane) & 7u;
#pragma unroll
        for (uint32_t g = 0; g < 4; ++g) {  // g = 2a + half: rows 16a + 8half + [0, 8)
          const uint32_t row = 8u * g + i;
          stmatrix_x4(buf + 64u * row + 16u * (m ^ ((row >> 1) & 3u)), h[4 * g], h[4 * g + 1], h[4 * g + 2],
                      h[4 * g + 3]);
        }
      } else {
        const uint32_t rb = buf + 64u * static_cast<uint32_t>(lane);
        const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
        for (uint32_t j = 0; j < 4; ++j)
          st_shared_v4(rb + 16u * (j ^ sw), h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
      }
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (to_slot) {
          if (row0 < p.w_rows) tma_store_3d(&p.tmap_w, buf, col0, row0, z);
        } else if (row0 < p.M) {
          tma_store_2d(&p.tmap_d, buf, col0, row0);
        }
        bulk_commit_group();  // one group per staged tile (possibly empty), so the waits above count tiles
      }
      ++epi_n;
    };
    auto store_tile16 = [&](int row0, int col0, const uint32_t(&h)[16]) { stage_tile(row0, col0, h, false, 0); };
    // The warp's 32 x 32 fp32 block at TMEM address t as two .16x256b.x4
    // loads (lanes +0 and +16), packed to 16-bit pairs in stmatrix order:
    // h[4g + j] = row 8g + lane/4, columns 8j + 2(lane%4) + {0, 1}.
    auto frag_load16 = [&](uint32_t t, uint32_t(&h)[16]) {
      uint32_t r0[16], r1[16];
      tmem_ld_16x256b_x4(t, r0);
      tmem_ld_16x256b_x4(t + (16u << 16), r1);
      tc_wait_ld();
      const bool bf = p.d_type == OUT_BF16;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          h[4 * hh + j] = bf ? pack_bf16(r0[4 * j + 2 * hh], r0[4 * j + 2 * hh + 1])
                             : pack_f16(r0[4 * j + 2 * hh], r0[4 * j + 2 * hh + 1]);
          h[8 + 4 * hh + j] = bf ? pack_bf16(r1[4 * j + 2 * hh], r1[4 * j + 2 * hh + 1])
                                 : pack_f16(r1[4 * j + 2 * hh], r1[4 * j + 2 * hh + 1]);
        }
    };
    // fragments only where they are staged for a TMA store of 16-bit values
    const bool frag16 = p.epi_frag && p.d_tma && p.d_type != OUT_F32 && !p.acc_f16;
    uint32_t tcount = 0;
    for (UnitCursor uc = uc_first; uc.valid; cursor_next(uc, num_clusters, p), ++tcount) {
      const int b = static_cast<int>(tcount % ACC);
      const uint32_t aph = (tcount / ACC) & 1u;
      if (!warp_wait(accf_bar(b), aph, wctx, SITE_EPI_ACC_FULL)) break;
      tc_fence_after();
      int mt, nt;
      tile_coords(uc.tile, p, mt, nt);
      const int row0 = mt * C::MMA_M + static_cast<int>(rank) * C::BM + 32 * q;
      const int row = row0 + lane;
      const int n0 = nt * BN;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * BN);
      auto release = [&]() {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CG == 2)
            mbar_arrive_cluster(mapa_shared(acce_bar(b), 0));
          else
            mbar_arrive(acce_bar(b));
        }
      };
      auto pack16 = [&](const uint32_t(&r)[32], uint32_t(&h)[16]) {
        if (p.d_type == OUT_BF16) {
#pragma unroll
          for (int k = 0; k < 16; ++k) h[k] = pack_bf16(r[2 * k], r[2 * k + 1]);
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) h[k] = pack_f16(r[2 * k], r[2 * k + 1]);
        }
      };
      if (uc.kb0 != 0 || uc.kb1 != p.num_k_blocks) {
        // part of a tile (split-K or stream-K): store this unit's fp32
        // partial into its own workspace slot (16-column halves of each
        // 32-column chunk through the staging tiles) and release the
        // accumulator; splitk_reduce_kernel, launched next on the stream,
        // sums each tile's slots in a fixed order into D.  Quadrants whose
        // rows all lie beyond M store nothing.
        if (row0 < p.M) {
          const int zslot = unit_slot(uc, cluster_id, p) * CG + static_cast<int>(rank);
#pragma unroll 1
          for (int c = part; c < BN / 32; c += nparts) {
            if (n0 + 32 * c >= p.N) break;
            uint32_t r[32];
            tmem_ld_32x32b_x32(tb + 32 * c, r);
            tc_wait_ld();
            uint32_t h[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) h[k] = r[k];
            stage_tile(32 * q, 32 * c, h, true, zslot);
#pragma unroll
            for (int k = 0; k < 16; ++k) h[k] = r[16 + k];
            stage_tile(32 * q, 32 * c + 16, h, true, zslot);
          }
        }
        release();
        continue;
      }
      if (early) {
        constexpr int HALF = (BN / 32 + 1) / 2;  // chunks per warp
        uint32_t h[HALF][16];
#pragma unroll
        for (int i = 0; i < HALF; ++i) {
          const int c = part + 2 * i;
          if (c < BN / 32) {
            if (p.acc_f16) {
              tmem_ld_32x32b_x16_pack16(tb + 32 * c, h[i]);
            } else if (frag16) {
              frag_load16(tb + 32 * c, h[i]);
            } else {
              uint32_t r[32];
              tmem_ld_32x32b_x32(tb + 32 * c, r);
              tc_wait_ld();
              pack16(r, h[i]);
            }
          }
        }
        tc_wait_ld();
        release();
#pragma unroll
        for (int i = 0; i < HALF; ++i) {
          const int c = part + 2 * i;
          if (c < BN / 32 && n0 + 32 * c < p.N) {
            if (p.d_tma)
              stage_tile(row0, n0 + 32 * c, h[i], false, 0, frag16);
            else if (row < p.M)
              store_row16(p, row, n0 + 32 * c, h[i]);
          }
        }
        continue;
      }
      if (p.acc_f16) {
#pragma unroll 1
        for (int c = part; c < BN / 32; c += nparts) {
          uint32_t h[16];
          tmem_ld_32x32b_x16_pack16(tb + 32 * c, h);
          tc_wait_ld();
          if (n0 + 32 * c < p.N) {
            if (p.d_tma)
              store_tile16(row0, n0 + 32 * c, h);
            else if (row < p.M)
              store_row16(p, row, n0 + 32 * c, h);
          }
        }
      } else if (frag16) {
#pragma unroll 1
        for (int c = part; c < BN / 32; c += nparts) {
          uint32_t h[16];
          frag_load16(tb + 32 * c, h);
          if (n0 + 32 * c < p.N) stage_tile(row0, n0 + 32 * c, h, false, 0, true);
        }
      } else {
#pragma unroll 1
        for (int c = part; c < BN / 32; c += nparts) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tb + 32 * c, r);
          tc_wait_ld();
          if (n0 + 32 * c < p.N) {
            if (TRANS && p.d_trans) {
              if (row < p.M) store_col32(p, row, n0 + 32 * c, r);
            } else if (p.d_tma && p.d_type == OUT_F32) {
              // fp32: two 16-column halves, each a 32 x 64-byte staging tile
              uint32_t h[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) h[k] = r[k];
              store_tile16(row0, n0 + 32 * c, h);
#pragma unroll
              for (int k = 0; k < 16; ++k) h[k] = r[16 + k];
              store_tile16(row0, n0 + 32 * c + 16, h);
            } else if (p.d_tma) {
              uint32_t h[16];
              pack16(r, h);
              store_tile16(row0, n0 + 32 * c, h);
            } else if (row < p.M) {
              store_row32(p, row, n0 + 32 * c, r);
            }
          }
        }
      }
      release();
    }
    // the staged tiles must be written out before the CTA ends
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
    if (warp == 4 && lane == 0) trace_stamp(p, TRACE_EPI_DONE);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  cta_barrier_unaligned();
  __syncwarp();
  if constexpr (CG == 2) cluster_sync();
  tc_fence_after();
  if (warp == 2) {
    tmem_dealloc<CG>(tmem_base, C::TMEM_COLS);
    if (lane == 0) trace_stamp_clock(p, TRACE_EXIT, TRACE_CLK_EXIT);
  }
}

}  // namespace tcg
