// Chained GEMM kernel: E = round(A . B1) . B2 for one CTA per 128 rows, the
// intermediate never leaving the SM.
//
//   phase 1  C = A . B1 into TMEM columns [0, N1) (fp32), tcgen05.mma with
//            both operands from 128B-swizzled shared tiles;
//   convert  the epilogue warps read C with tcgen05.ld, round it to the
//            operand type and write it back with tcgen05.st as 16-bit pairs
//            at columns [0, N1/2): row m in lane m, K element k of the second
//            product in column k/2 -- the layout an A operand in tensor memory
//            has ("tcgen05.mma" page, "Operands and repeat axes": A from
//            "Shared or TMEM"; the layout pinned by the TMEM-A probe);
//   phase 2  for each 192-column tile of E: N1/16 tcgen05.mma with A read
//            from TMEM column 8*step and B2 from shared memory (stages of
//            128 of N1, two tiles' worth in flight for N1 = 256), into one of
//            two accumulators (columns 128 and 320), drained by the epilogue
//            while the other fills.
//
// Warp roles as in the main kernel: warp 0 TMA producer (one ring for both
// phases), warp 1 MMA issuer, warp 2 TMEM allocation, warp 3 barrier set-up,
// warps 4..11 epilogue (two per TMEM lane quadrant).  Work units are (128-row
// tile, group of E tiles); with fewer row tiles than SMs the E tiles are
// split into groups and each group's unit recomputes its C.
//
// Clusters of CS CTAs (CS = 1 or 2) take CS neighbouring row tiles of the
// same group, so they walk the same B1 / B2 tiles in the same order: each CTA
// loads 1/CS of every B tile and multicasts it into the same stage of all CS
// CTAs, which cuts the B bytes an SM pulls from L2 by CS.  The MMAs stay
// cta_group::1 (every CTA issues its own from its own shared memory and
// TMEM); a stage is refilled once all CS CTAs' MMAs have read it (each MMA
// warp's commit arrives on the empty barrier of every CTA in the cluster).
// Every wait is bounded; a timeout records an error word and the CTA drains
// and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.h"
#include "gemm_chain.cuh"
#include "gemm_kernel.cuh"
#include "tmem_ldst.cuh"

namespace tcg {

namespace {

constexpr uint32_t CHAIN_A_BYTES = 128 * 128;            // one 128-row x 64-element stage of A
constexpr uint32_t CHAIN_B2_BOX_BYTES = CHAIN_BN2 * 128;  // one CHAIN_BN2-row x 64-element box of B2
static_assert(2 * CHAIN_B2_BOX_BYTES <= CHAIN_STAGE_BYTES, "two B2 boxes per stage");

template <int CS>
__global__ void __launch_bounds__(CHAIN_THREADS, 1) gemm_chain_kernel(const __grid_constant__ ChainParams p) {
  // trace: globaltimer and the SM cycle counter read back to back
  auto trace_clock = [&](int slot, int clk_slot) {
    if (p.trace && static_cast<int>(blockIdx.x) < p.trace_ctas) {
      const uint64_t t = globaltimer();
      const uint64_t c = clock64();
      p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + slot] = t;
      p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + clk_slot] = c;
    }
  };
  if (threadIdx.x == 0) trace_clock(TRACE_ENTRY, TRACE_CLK_ENTRY);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + CHAIN_BAR_OFF;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (CHAIN_STAGES + s); };
  const uint32_t c_full = bar0 + 8u * (2 * CHAIN_STAGES);
  const uint32_t a2_ready = c_full + 8u;
  const uint32_t conv_mid = c_full + 16u;
  auto d_full = [&](uint32_t b) { return c_full + 24u + 8u * b; };
  auto d_empty = [&](uint32_t b) { return c_full + 40u + 8u * b; };
  const uint32_t drain_bar = c_full + 56u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + CHAIN_BAR_OFF + 8 * CHAIN_NUM_BARS);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const WaitCtx wctx{p.timeout_ns, p.err, abort_flag};
  const uint32_t rank = CS > 1 ? cluster_ctarank() : 0u;
  const int cluster_id = blockIdx.x / CS;
  const int num_clusters = gridDim.x / CS;
  constexpr uint16_t CLUSTER_MASK = static_cast<uint16_t>((1u << CS) - 1u);

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&p.tmap_a);
    prefetch_tmap(&p.tmap_b1);
    prefetch_tmap(&p.tmap_b2);
    prefetch_tmap(&p.tmap_e);
  }
  if (threadIdx.x == 96) {
    for (int s = 0; s < CHAIN_STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), CS);  // one commit from each CTA's MMA warp
    }
    mbar_init(c_full, 1);
    mbar_init(a2_ready, CHAIN_EPI_WARPS);
    mbar_init(conv_mid, CHAIN_EPI_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(d_full(b), 1);
      mbar_init(d_empty(b), CHAIN_EPI_WARPS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbarrier_init();
  }
  if (warp == 2) {
    tmem_alloc<1>(smem_u32(tmem_slot), 512);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (CS > 1) cluster_sync();  // peers' barriers are initialised before any multicast
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // cluster unit u: this CTA's row tile CS * (u % m_blocks) + rank (past
  // the last tile for some CTAs of the last block: those load zero-filled A,
  // keep the cluster's B multicasts going and store nothing), E tiles
  // [t0, t1) of group u / m_blocks
  auto unit_tiles = [&](int u, int& mt, int& t0, int& t1) {
    mt = CS * (u % p.m_blocks) + static_cast<int>(rank);
    t0 = (u / p.m_blocks) * p.tiles_per_group;
    t1 = min(p.n2_tiles, t0 + p.tiles_per_group);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, s = 0, ph = 0;
    bool ok = true;
    for (int u = cluster_id; u < p.num_units && ok; u += num_clusters) {
      int mt, t0, t1;
      unit_tiles(u, mt, t0, t1);
      const int stages = p.k1_blocks + (t1 - t0) * p.k2_blocks;
      const int m0 = 128 * mt;
      for (int i = 0; i < stages; ++i) {
        if (!wait_uniform(empty_bar(s), ph ^ 1u, wctx, SITE_PROD_EMPTY)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          // this stage's full barrier counts the whole tile: this CTA's A,
          // plus every CTA's slice of B (this one's own included)
          const uint32_t sa = sbase + s * CHAIN_STAGE_BYTES;
          auto load_b = [&](uint32_t dst, const CUtensorMap* map, int x, int y) {
            if constexpr (CS > 1)
              tma_load_2d_multicast(dst, map, x, y, full_bar(s), CLUSTER_MASK);
            else
              tma_load_2d(dst, map, x, y, full_bar(s));
          };
          if (i < p.k1_blocks) {
            const int rows = p.N1 / CS;
            mbar_arrive_expect_tx(full_bar(s), CHAIN_A_BYTES + static_cast<uint32_t>(p.N1) * 128u);
            tma_load_2d(sa, &p.tmap_a, 64 * i, m0, full_bar(s));
            load_b(sa + CHAIN_A_BYTES + static_cast<uint32_t>(rank * rows) * 128u, &p.tmap_b1, 64 * i,
                   static_cast<int>(rank) * rows);
          } else {
            // a second-product stage holds up to two 64-column boxes of the
            // E tile's B2 rows (128 of N1), so that the ring keeps two
            // tiles' B2 in flight
            const int j = i - p.k1_blocks;
            const int t = t0 + j / p.k2_blocks;
            const int x0 = 128 * (j % p.k2_blocks);
            const uint32_t boxes = x0 + 64 < p.N1 ? 2u : 1u;
            constexpr int rows = CHAIN_BN2 / CS;
            mbar_arrive_expect_tx(full_bar(s), boxes * CHAIN_BN2 * 128u);
            for (uint32_t bx = 0; bx < boxes; ++bx)
              load_b(sa + bx * CHAIN_B2_BOX_BYTES + rank * rows * 128u, &p.tmap_b2, x0 + 64 * static_cast<int>(bx),
                     CHAIN_BN2 * t + static_cast<int>(rank) * rows);
          }
        }
        __syncwarp();
        ++it;
        if (++s == CHAIN_STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && elect_one()) {
      // let the copies in flight land before the CTA can exit
      const uint32_t n_out = it < static_cast<uint32_t>(CHAIN_STAGES) ? it : static_cast<uint32_t>(CHAIN_STAGES);
      for (uint32_t j = it - n_out; j < it; ++j) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(full_bar(j % CHAIN_STAGES), (j / CHAIN_STAGES) & 1u) &&
               globaltimer() - t0 < 20000000ull) {
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint64_t hi = sdesc_hi(16, 1024, SW_128B);
    // stage s has been read by this CTA's MMAs: tell every CTA whose
    // multicast refills it
    auto release = [&](uint32_t s) {
      if constexpr (CS > 1)
        tc_commit_multicast(empty_bar(s), CLUSTER_MASK);
      else
        tc_commit<1>(empty_bar(s));
    };
    uint32_t s = 0, ph = 0, dt = 0, uc = 0;
    bool ok = true;
    for (int u = cluster_id; u < p.num_units && ok; u += num_clusters, ++uc) {
      int mt, t0, t1;
      unit_tiles(u, mt, t0, t1);
      // C (fp32) overlaps the first accumulator and its 16-bit copy is read
      // by the previous unit's second product: both accumulators must have
      // been drained (which follows their last MMAs' completion)
      for (uint32_t back = 1; back <= 2 && ok; ++back) {
        if (dt < back) break;
        const uint32_t t = dt - back;
        if (!wait_uniform(d_empty(t & 1u), (t >> 1) & 1u, wctx, SITE_MMA_ACC_EMPTY)) ok = false;
      }
      if (!ok) break;
      tc_fence_after();
      for (int kb = 0; kb < p.k1_blocks; ++kb) {
        if (!wait_uniform(full_bar(s), ph, wctx, SITE_MMA_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sa = sbase + s * CHAIN_STAGE_BYTES;
          const uint64_t ad = sdesc(sa, hi), bd = sdesc(sa + CHAIN_A_BYTES, hi);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // 16 K elements = 32 bytes = 2 descriptor units per step
            mma_f16<1>(tmem_base, ad + 2 * j, bd + 2 * j, p.idesc1, (kb | j) ? 1u : 0u);
          release(s);
        }
        __syncwarp();
        if (++s == CHAIN_STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit<1>(c_full);
      __syncwarp();
      // the epilogue has rewritten C as the 16-bit A operand
      if (!wait_uniform(a2_ready, uc & 1u, wctx, SITE_MMA_FULL)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int t = t0; t < t1 && ok; ++t, ++dt) {
        const uint32_t b = dt & 1u;
        if (!wait_uniform(d_empty(b), ((dt >> 1) & 1u) ^ 1u, wctx, SITE_MMA_ACC_EMPTY)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + CHAIN_D_COL0 + CHAIN_BN2 * b;
        for (int kb = 0; kb < p.k2_blocks; ++kb) {
          if (!wait_uniform(full_bar(s), ph, wctx, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sa = sbase + s * CHAIN_STAGE_BYTES;
            const uint64_t bd0 = sdesc(sa, hi), bd1 = sdesc(sa + CHAIN_B2_BOX_BYTES, hi);
#pragma unroll
            for (int j = 0; j < 8; ++j) {  // 16 of N1 per MMA, four per 64-column box
              const int step = 8 * kb + j;
              if (step < p.k2_steps)
                mma_f16_tmem_a(d_tmem, tmem_base + 8u * static_cast<uint32_t>(step), (j < 4 ? bd0 : bd1) + 2 * (j & 3),
                               p.idesc2, step ? 1u : 0u);
            }
            release(s);
          }
          __syncwarp();
          if (++s == CHAIN_STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (elect_one()) tc_commit<1>(d_full(b));
        __syncwarp();
      }
    }
    if (lane == 0 && p.trace && static_cast<int>(blockIdx.x) < p.trace_ctas)
      p.trace[static_cast<int64_t>(blockIdx.x) * TRACE_SLOTS + TRACE_UNITS] = uc;
    if (!ok && elect_one()) {
      tc_commit<1>(drain_bar);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < 20000000ull) {
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;           // TMEM lane quadrant
    const int part = (warp - 4) >> 2;  // 0 or 1: which half of the columns
    const uint32_t lanes = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
    const uint32_t buf0 = sbase + CHAIN_EPI_OFF + static_cast<uint32_t>((warp - 4) * CHAIN_EPI_BUFS * 32 * 64);
    const bool bf = p.in_bf16 != 0;
    uint32_t dt = 0, uc = 0, stores = 0;
    bool ok = true;
    // one 32-row x 64-byte tile of E at (row0, col0) through the staging buffer
    auto stage = [&](int row0, int col0, const uint32_t* h) {
      const uint32_t buf = buf0 + (stores % CHAIN_EPI_BUFS) * 32u * 64u;
      if (stores >= static_cast<uint32_t>(CHAIN_EPI_BUFS)) {
        if (lane == 0) bulk_wait_group_read<CHAIN_EPI_BUFS - 1>();  // this buffer's last store has read it
        __syncwarp();
      }
      const uint32_t rb = buf + 64u * static_cast<uint32_t>(lane);
      const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
      for (uint32_t j = 0; j < 4; ++j) st_shared_v4(rb + 16u * (j ^ sw), h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(&p.tmap_e, buf, col0, row0);
        bulk_commit_group();
      }
      ++stores;
    };
    for (int u = cluster_id; u < p.num_units && ok; u += num_clusters, ++uc) {
      int mt, t0, t1;
      unit_tiles(u, mt, t0, t1);
      const int row0 = 128 * mt + 32 * q;
      // ---- C (fp32) -> 16-bit pairs in place.  This warp reads C columns
      // [128*part, 128*part + 128) of its 32 lanes; the other warp of the
      // quadrant writes into that range, so every read lands before any write
      // (conv_mid), then each writes its packed words.
      if (!warp_wait(c_full, uc & 1u, wctx, SITE_EPI_ACC_FULL)) break;
      tc_fence_after();
      uint32_t packed[4][16];
#pragma unroll
      for (int c = 0; c < 4; c += 2) {  // two loads in flight per wait
        const int col = 128 * part + 32 * c;
        uint32_t r[2][32];
        if (col < p.N1) tmem_ld_32x32b_x32(lanes + static_cast<uint32_t>(col), r[0]);
        if (col + 32 < p.N1) tmem_ld_32x32b_x32(lanes + static_cast<uint32_t>(col + 32), r[1]);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int k = 0; k < 16; ++k)
            packed[c + i][k] = bf ? pack_bf16(r[i][2 * k], r[i][2 * k + 1]) : pack_f16(r[i][2 * k], r[i][2 * k + 1]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(conv_mid);
      if (!warp_wait(conv_mid, uc & 1u, wctx, SITE_EPI_ACC_FULL)) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = 128 * part + 32 * c;
        // columns past N1 (a multiple of 16) are never read by the MMAs
        if (col < p.N1) stx_32x32b_x16(lanes + static_cast<uint32_t>(col / 2), packed[c]);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(a2_ready);
      // ---- E tiles
      for (int t = t0; t < t1; ++t, ++dt) {
        const uint32_t b = dt & 1u;
        if (!warp_wait(d_full(b), (dt >> 1) & 1u, wctx, SITE_EPI_ACC_FULL)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dcol = CHAIN_D_COL0 + CHAIN_BN2 * b;
        // this warp's three 32-column chunks (part, part + 2, part + 4): two
        // loads in flight, their stores, the third load, then the
        // accumulator is released before the third store
        static_assert(CHAIN_BN2 == 192, "three chunks per epilogue warp");
        const int n0 = CHAIN_BN2 * t + 32 * part;
        auto store_chunk = [&](int col0, const uint32_t* r) {
          if (row0 >= p.M || col0 >= p.N2) return;  // the map clips the rest of a ragged tile
          if (p.e_type == OUT_F32) {
            stage(row0, col0, r);
            stage(row0, col0 + 16, r + 16);
          } else {
            uint32_t h[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              h[k] = p.e_type == OUT_BF16 ? pack_bf16(r[2 * k], r[2 * k + 1]) : pack_f16(r[2 * k], r[2 * k + 1]);
            stage(row0, col0, h);
          }
        };
        {
          uint32_t r[2][32];
          tmem_ld_32x32b_x32(lanes + dcol + 32u * part, r[0]);
          tmem_ld_32x32b_x32(lanes + dcol + 32u * (part + 2), r[1]);
          tc_wait_ld();
          store_chunk(n0, r[0]);
          store_chunk(n0 + 64, r[1]);
        }
        uint32_t r[32];
        tmem_ld_32x32b_x32(lanes + dcol + 32u * (part + 4), r);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(d_empty(b));
        store_chunk(n0 + 128, r);
      }
    }
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  cta_barrier_unaligned();
  __syncwarp();
  if constexpr (CS > 1) cluster_sync();  // no peer multicasts into this CTA or arrives on its barriers any more
  tc_fence_after();
  if (warp == 2) {
    tmem_dealloc<1>(tmem_base, 512);
    if (lane == 0) trace_clock(TRACE_EXIT, TRACE_CLK_EXIT);
  }
}

}  // namespace

KernelInfo kinfo_chain(int cluster) {
  const void* fn = cluster == 2 ? reinterpret_cast<const void*>(&gemm_chain_kernel<2>)
                                : reinterpret_cast<const void*>(&gemm_chain_kernel<1>);
  return KernelInfo{fn, CHAIN_SMEM_BYTES, cluster == 2 ? 2 : 1, CHAIN_BN2, KIND_F16, CHAIN_THREADS};
}

// The shared-memory attribute was set when the cluster capacity was queried
// (max_clusters_for on the host side, once per device and variant), so that
// calls captured into a CUDA graph make no attribute call.
cudaError_t launch_chain(const ChainParams& p, int cluster, int grid, cudaStream_t s) {
  const KernelInfo ki = kinfo_chain(cluster);
  if (ki.cta_group != cluster) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(CHAIN_THREADS, 1, 1);
  cfg.dynamicSmemBytes = CHAIN_SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cluster;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = cluster > 1 ? 1 : 0;
  void* args[] = {const_cast<ChainParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, ki.func, args);
}

}  // namespace tcg
