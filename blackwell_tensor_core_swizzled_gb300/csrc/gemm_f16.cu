// kind::f16 GEMM variants (f16 and bf16 operands, f32 or f16 accumulation).
//   cta_group::1: 128 x 256 tile per CTA, 4-stage ring, 2 TMEM accumulators.
//   cta_group::2: 256 x 256 tile per CTA pair (each CTA stages its 128 rows of
//                 A and 128 rows of B), 6-stage ring, 2 accumulators.
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {


KernelInfo kinfo_f16(int cta_group, bool skinny) {
  if (skinny) {
    // M <= 32, single CTA, K-major A: 64-column tiles (more CTAs), 32 staged
    // A rows, 16-stage ring (twice the B bytes in flight per SM)
    using C = GemmCfg<1, 64, 2, 16, KIND_F16, 32>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 64, 2, 16, KIND_F16, 32>), C::SMEM_BYTES, 1, 64,
            KIND_F16, C::THREADS};
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
