// Internal host-side interface shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tcg.h"

namespace tcg {

struct GemmParams;

// One compiled GEMM kernel variant.
struct KernelInfo {
  const void* func;  // host stub of the __global__ function
  int smem_bytes;    // dynamic shared memory it needs
  int cta_group;     // 1 or 2 (cluster of 2 CTAs)
  int bn;            // accumulator columns (N tile)
  int kind;          // Kind
  int threads;
};

// Variant getters (one per translation unit that instantiates kernels).
enum F16Variant {
  F16_WIDE = 0, F16_SKINNY_M = 1, F16_NARROW_N = 2, F16_SKINNY_M64 = 3, F16_SKINNY_M128 = 4, F16_PAIR_N128 = 5
};
KernelInfo kinfo_f16(int cta_group, F16Variant v = F16_WIDE);
KernelInfo kinfo_tf32(int cta_group);
KernelInfo kinfo_mxf8(int cta_group);  // BN 256, one accumulator (single CTA or CTA pair)
// packed FP4: kind::mxf4 (scale_vec::2X, e8m0) or kind::mxf4nvf4 (scale_vec::4X,
// UE4M3); wide: CTA pairs with 256 x 384 tiles (two MMAs per K step), K-major B
KernelInfo kinfo_fp4(int cta_group, bool nvf4, bool wide = false);

// How a block-scaled format's scales are staged: K elements per scale, K
// steps (of four scales per row, one 512-byte chunk per 128 rows) per ring
// stage, and the byte that stands for a scale of one.
struct ScaleFormat {
  int block;
  int kch;
  uint32_t fill;
};
ScaleFormat scale_format(tcg_input t);
// Bytes of the scale image of `rows` rows and K elements, tiles of tile_rows.
int64_t sf_image_bytes_fmt(tcg_input t, int64_t rows, int64_t K, int tile_rows);
// Scale-factor rearrangement kernel launch (gemm_mxf8.cu).
cudaError_t launch_sf_prepare(tcg_input t, const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint8_t* img,
                              cudaStream_t stream);
// Both operands' images in one launch.
cudaError_t launch_sf_prepare_pair(tcg_input t, const uint8_t* sfa, int64_t rows_a, int tile_a, uint8_t* img_a,
                                   const uint8_t* sfb, int64_t rows_b, int tile_b, uint8_t* img_b, int64_t K,
                                   cudaStream_t stream);

// Sum of the partial-tile slots of a split-K / stream-K GEMM into D
// (splitk_reduce.cu); launched after the GEMM on the same stream.
cudaError_t launch_splitk_reduce(const GemmParams& p, int cg, int num_clusters, cudaStream_t stream);

// Chained GEMM kernel launch (gemm_chain.cu).
struct ChainParams;
// The chained kernel for clusters of `cluster` CTAs (1 or 2) sharing B
// tiles by multicast (gemm_chain.cu); KernelInfo::cta_group carries the
// cluster size.
KernelInfo kinfo_chain(int cluster);
cudaError_t launch_chain(const ChainParams& p, int cluster, int grid, cudaStream_t stream);

// Host state helpers (api.cu).
int record_cuda(cudaError_t e);              // stores the message, returns TCG_ERR_CUDA (or TCG_OK)
int current_device_checked(int* dev);        // TCG_OK if the current device is usable sm_103
unsigned long long* device_error_word(int dev);
uint64_t wait_timeout_ns();
void set_launch_count(int n);

}  // namespace tcg

namespace tcg {
// Sets the text tcg_last_error_string() returns on this thread.
void set_error_message(const char* msg);
}  // namespace tcg
