// kind::f16 GEMM variants (f16 and bf16 operands, f32 or f16 accumulation).
//   cta_group::1: 128 x 256 tile per CTA, 4-stage ring, 2 TMEM accumulators.
//   cta_group::2: 256 x 256 tile per CTA pair (each CTA stages its 128 rows of
//                 A and 128 rows of B), 6-stage ring, 2 accumulators.
//   skinny M:     128 x 64 tiles staging 32 / 64 / 128 rows of A (M <= 32 /
//                 64 / 128), 16- / 12- / 8-stage rings.
//   narrow N:     128 x 32 tiles, 10-stage ring.
//   pair N128:    256 x 128 pair tiles, 8-stage ring (few pair tiles).
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {


KernelInfo kinfo_f16(int cta_group, F16Variant v) {
  if (v == F16_SKINNY_M) {
    // M <= 32, single CTA, K-major A: 64-column tiles (more CTAs), 32 staged
    // A rows, 16-stage ring (twice the B bytes in flight per SM)
    using C = GemmCfg<1, 64, 2, 16, KIND_F16, 32>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 64, 2, 16, KIND_F16, 32>), C::SMEM_BYTES, 1, 64,
            KIND_F16, C::THREADS};
  }
  if (v == F16_SKINNY_M64) {
    // 32 < M <= 64: the same 64-column tiles with 64 staged A rows, 12 stages
    using C = GemmCfg<1, 64, 2, 12, KIND_F16, 64>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 64, 2, 12, KIND_F16, 64>), C::SMEM_BYTES, 1, 64,
            KIND_F16, C::THREADS};
  }
  if (v == F16_SKINNY_M128) {
    // 64 < M <= 128: 64-column tiles over the full 128-row A tile, 8 stages
    using C = GemmCfg<1, 64, 2, 8, KIND_F16>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 64, 2, 8, KIND_F16>), C::SMEM_BYTES, 1, 64, KIND_F16,
            C::THREADS};
  }
  if (v == F16_NARROW_N) {
    // N <= 32 (and few-row problems computed transposed), single CTA:
    // 128 x 32 tiles, 10-stage ring of 16 KB A + 4 KB B stages
    using C = GemmCfg<1, 32, 2, 10, KIND_F16>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 32, 2, 10, KIND_F16>), C::SMEM_BYTES, 1, 32, KIND_F16,
            C::THREADS};
  }
  if (v == F16_PAIR_N128) {
    // few pair tiles: 256 x 128 pair tiles (twice as many), 8 stages
    using C = GemmCfg<2, 128, 2, 8, KIND_F16>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 128, 2, 8, KIND_F16>), C::SMEM_BYTES, 2, 128, KIND_F16,
            C::THREADS};
  }
  if (cta_group == 2) {
    using C = GemmCfg<2, 256, 2, 6, KIND_F16>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 256, 2, 6, KIND_F16>), C::SMEM_BYTES, 2, 256,
            KIND_F16, C::THREADS};
  }
  using C = GemmCfg<1, 256, 2, 4, KIND_F16>;
  return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 2, 4, KIND_F16>), C::SMEM_BYTES, 1, 256, KIND_F16,
          C::THREADS};
}

}  // namespace tcg
