// Chained GEMM E = round(A . B1) . B2 with the intermediate kept in tensor
// memory as the second product's A operand ("tcgen05.mma" page, "Operands and
// repeat axes": A may come from shared memory or TMEM).  Parameters shared by
// the kernel (gemm_chain.cu) and the host entry point (api.cu).
#pragma once

#include <cuda.h>

#include <cstdint>

namespace tcg {

struct ChainParams {
  CUtensorMap tmap_a;   // A [M][K], 64-element x 128-row boxes, 128-byte swizzle
  CUtensorMap tmap_b1;  // B1 [N1][K], 64-element x N1-row boxes
  CUtensorMap tmap_b2;  // B2 [N2][N1], 64-element x CHAIN_BN2-row boxes
  CUtensorMap tmap_e;   // E [M][N2], 32-row x 64-byte boxes, 64-byte swizzle
  int M, N1, N2, K;
  int m_tiles;          // 128-row tiles of A / E
  int m_blocks;         // cluster-sized blocks of row tiles: cdiv(m_tiles, cluster size)
  int n2_tiles;         // CHAIN_BN2-column tiles of E
  int tiles_per_group;  // E tiles one unit computes
  int num_units;        // m_blocks x groups; cluster unit u -> (block u % m_blocks, group u / m_blocks)
  int k1_blocks;        // ring stages of the first product (64 K each)
  int k2_blocks;        // ring stages per E tile of the second product (128 of N1 each)
  int k2_steps;         // second-product MMAs: N1 / 16
  uint32_t idesc1, idesc2;
  int in_bf16;          // operand type (and the intermediate's): bf16, else f16
  int e_type;           // OutType of E
  unsigned long long* err;
  uint64_t timeout_ns;
  // optional trace (null: off), the GEMM kernel's slot layout: per CTA
  // globaltimer at entry (0) and exit (6), units computed (7), and the SM
  // cycle counter next to the two stamps (8, 9)
  unsigned long long* trace;
  int trace_ctas;
};

// E tiles of 192 columns in two accumulators at TMEM columns 128 and 320,
// beside the 16-bit A operand at [0, N1/2) (the intermediate C, fp32 at
// [0, N1), is rewritten there in place; while it is fp32 it overlaps the
// first accumulator, so a row tile's first product starts once the previous
// tile's accumulators are drained)
constexpr int CHAIN_BN2 = 192;
constexpr int CHAIN_D_COL0 = 128;
constexpr int CHAIN_STAGES = 4;
constexpr int CHAIN_STAGE_BYTES = 48 * 1024;  // A (16 KiB) + B1 (up to 256 rows, 32 KiB), or two B2 boxes
constexpr int CHAIN_EPI_WARPS = 8;
constexpr int CHAIN_THREADS = 32 * (4 + CHAIN_EPI_WARPS);
// per epilogue warp, CHAIN_EPI_BUFS staging tiles of 32 rows x 64 bytes: a
// tile is rewritten only once the store before the last has read it
constexpr int CHAIN_EPI_BUFS = 2;
constexpr int CHAIN_EPI_OFF = CHAIN_STAGES * CHAIN_STAGE_BYTES;
constexpr int CHAIN_BAR_OFF = CHAIN_EPI_OFF + CHAIN_EPI_WARPS * CHAIN_EPI_BUFS * 32 * 64;
// full[S], empty[S], c_full, a2_ready, conv_mid, d_full[2], d_empty[2], drain
constexpr int CHAIN_NUM_BARS = 2 * CHAIN_STAGES + 8;
constexpr int CHAIN_SMEM_BYTES = 1024 + CHAIN_BAR_OFF + CHAIN_NUM_BARS * 8 + 16;
static_assert(CHAIN_SMEM_BYTES <= 232448, "dynamic shared memory");

}  // namespace tcg
