// Block-scaled MXFP8 GEMM variants (kind::mxf8f6f4.block_scale.scale_vec::1X,
// E4M3 operands, one e8m0 scale per 32 K elements) and the scale-factor
// rearrangement kernel.
//
// TMEM budget (128 lanes x 512 columns, "tcgen05.cp" page, "TMEM shape and
// replicas"): the CTA-pair variant keeps two 224-column accumulators (448
// columns) and four 16-column scale slots; the single-CTA variant one
// 256-column accumulator and four scale slots.
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {


KernelInfo kinfo_mxf8(int cta_group) {
  if (cta_group == 2) {
    using C = GemmCfg<2, 224, 2, 6, KIND_MXF8>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 224, 2, 6, KIND_MXF8>), C::SMEM_BYTES, 2, 224,
            KIND_MXF8, C::THREADS};
  }
  using C = GemmCfg<1, 256, 1, 4, KIND_MXF8>;
  return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 1, 4, KIND_MXF8>), C::SMEM_BYTES, 1, 256,
          KIND_MXF8, C::THREADS};
}

// Rearranges plain row-major e8m0 scales sf[rows][kblocks] into the image the
// GEMM streams: for every K step of four scale blocks and every tile of
// tile_rows rows, ceil(tile_rows/128) chunks of 512 bytes in which the scale
// of tile row r and block kb sits at byte 16*(r%32) + 4*(r//32) + kb.  One
// tcgen05.cp .32x128b.warpx4 of such a chunk (source row i = bytes
// [16i, 16i+16)) puts it at TMEM lane r%32 (and its three replicas),
// byte-column 4*(r//32)+kb, which is where the "tcgen05.mma" page places
// block scales.  Each thread writes one 32-bit word: the four K blocks of one
// row, which are contiguous in the plain layout.  Absent rows / blocks get
// 127 (a scale of one).
__global__ void sf_prepare_kernel(const uint8_t* __restrict__ sf, int64_t rows, int64_t kblocks, int tile_rows,
                                  int64_t tiles, int chunks, int64_t total_words, uint32_t* __restrict__ img) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total_words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int w = static_cast<int>(i & 127);
    int64_t chunk_id = i >> 7;
    const int c = static_cast<int>(chunk_id % chunks);
    chunk_id /= chunks;
    const int64_t t = chunk_id % tiles;
    const int64_t ks = chunk_id / tiles;
    const int rl = c * 128 + 32 * (w & 3) + (w >> 2);
    const int64_t r = t * tile_rows + rl;
    uint32_t v = 0x7F7F7F7Fu;
    if (rl < tile_rows && r < rows) {
      v = 0u;
#pragma unroll
      for (int kb = 0; kb < 4; ++kb) {
        const int64_t kk = ks * 4 + kb;
        const uint32_t b = kk < kblocks ? static_cast<uint32_t>(sf[r * kblocks + kk]) : 127u;
        v |= b << (8 * kb);
      }
    }
    img[i] = v;
  }
}

cudaError_t launch_sf_prepare(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint8_t* img,
                              cudaStream_t stream) {
  const int64_t kblocks = (K + 31) / 32;
  const int64_t ksteps = (kblocks + 3) / 4;
  const int64_t tiles = (rows + tile_rows - 1) / tile_rows;
  const int chunks = (tile_rows + 127) / 128;
  const int64_t total_words = ksteps * tiles * chunks * 128;
  if (total_words == 0) return cudaSuccess;
  int64_t blocks = (total_words + 255) / 256;
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  sf_prepare_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(sf, rows, kblocks, tile_rows, tiles, chunks,
                                                                        total_words, reinterpret_cast<uint32_t*>(img));
  return cudaGetLastError();
}

}  // namespace tcg
