// kind::tf32 GEMM variants (float32 storage read as TF32, f32 accumulation).
// Same tiling as the kind::f16 variants; a ring stage holds 32 K elements
// (one 128-byte swizzle row) and each stage is four K=8 MMA issues.
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {


KernelInfo kinfo_tf32(int cta_group) {
  if (cta_group == 2) {
    using C = GemmCfg<2, 256, 2, 6, KIND_TF32>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 256, 2, 6, KIND_TF32>), C::SMEM_BYTES, 2, 256,
            KIND_TF32, C::THREADS};
  }
  using C = GemmCfg<1, 256, 2, 4, KIND_TF32>;
  return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 2, 4, KIND_TF32>), C::SMEM_BYTES, 1, 256,
          KIND_TF32, C::THREADS};
}

}  // namespace tcg
