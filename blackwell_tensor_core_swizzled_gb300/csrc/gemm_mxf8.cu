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
// block scales; the scale warps write the same placement with tcgen05.st.
// Absent rows / blocks get 127 (a scale of one).
//
// One block per (128-row chunk of one matrix, SF_KS_CHUNK K steps); SFA and
// SFB go in the same launch.  The four scale bytes of one row and K step are
// contiguous in the plain layout, so each output word is one 32-bit word of
// the input: the block reads its rows' words (consecutive threads, consecutive
// words of a row) into shared memory and writes each K step's 512-byte chunk
// as 128 consecutive words.  When the row stride is not a multiple of four
// bytes (K not a multiple of 128) or the base is misaligned, the words are
// assembled from bytes instead.
struct SfJob {
  const uint8_t* sf;
  int64_t rows;
  int64_t tiles;
  int tile_rows;
  int chunks;
  uint32_t* img;
};

constexpr int SF_KS_CHUNK = 32;

__global__ void __launch_bounds__(256) sf_prepare_kernel(SfJob ja, SfJob jb, int64_t kblocks, int64_t ksteps,
                                                         int64_t kparts) {
  __shared__ uint32_t words[128][SF_KS_CHUNK + 1];
  int64_t blk = blockIdx.x / kparts;
  const int64_t kp = blockIdx.x % kparts;
  const int64_t na = ja.tiles * ja.chunks;
  const SfJob j = blk < na ? ja : jb;
  if (blk >= na) blk -= na;
  const int64_t t = blk / j.chunks;
  const int c = static_cast<int>(blk % j.chunks);
  const int64_t row0 = t * j.tile_rows + 128 * c;
  const int valid = static_cast<int>(
      max(static_cast<int64_t>(0), min(min(static_cast<int64_t>(j.tile_rows) - 128 * c, j.rows - row0),
                                       static_cast<int64_t>(128))));
  const int64_t ks0 = kp * SF_KS_CHUNK;
  const int nks = static_cast<int>(min(static_cast<int64_t>(SF_KS_CHUNK), ksteps - ks0));
  const bool word_loads = (kblocks % 4 == 0) && (reinterpret_cast<uintptr_t>(j.sf) % 4 == 0);
  for (int i = threadIdx.x; i < 128 * SF_KS_CHUNK; i += blockDim.x) {
    const int rl = i / SF_KS_CHUNK, kw = i % SF_KS_CHUNK;
    uint32_t v = 0x7F7F7F7Fu;
    if (rl < valid && kw < nks) {
      const uint8_t* src = j.sf + (row0 + rl) * kblocks + 4 * (ks0 + kw);
      if (word_loads) {
        v = *reinterpret_cast<const uint32_t*>(src);
      } else {
        v = 0u;
        for (int b = 0; b < 4; ++b) {
          const uint32_t byte = 4 * (ks0 + kw) + b < kblocks ? static_cast<uint32_t>(src[b]) : 127u;
          v |= byte << (8 * b);
        }
      }
    }
    words[rl][kw] = v;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < nks * 128; i += blockDim.x) {
    const int ksl = i >> 7, w = i & 127;
    const int rl = 32 * (w & 3) + (w >> 2);
    j.img[(((ks0 + ksl) * j.tiles + t) * j.chunks + c) * 128 + w] = words[rl][ksl];
  }
}

namespace {
SfJob make_job(const uint8_t* sf, int64_t rows, int tile_rows, uint8_t* img) {
  SfJob j;
  j.sf = sf;
  j.rows = rows;
  j.tile_rows = tile_rows;
  j.tiles = sf ? (rows + tile_rows - 1) / tile_rows : 0;
  j.chunks = (tile_rows + 127) / 128;
  j.img = reinterpret_cast<uint32_t*>(img);
  return j;
}
}  // namespace

cudaError_t launch_sf_prepare_pair(const uint8_t* sfa, int64_t rows_a, int tile_a, uint8_t* img_a,
                                   const uint8_t* sfb, int64_t rows_b, int tile_b, uint8_t* img_b, int64_t K,
                                   cudaStream_t stream) {
  const int64_t kblocks = (K + 31) / 32;
  const int64_t ksteps = (kblocks + 3) / 4;
  const int64_t kparts = (ksteps + SF_KS_CHUNK - 1) / SF_KS_CHUNK;
  const SfJob ja = make_job(sfa, rows_a, tile_a, img_a);
  const SfJob jb = make_job(sfb, rows_b, tile_b, img_b);
  const int64_t blocks = (ja.tiles * ja.chunks + jb.tiles * jb.chunks) * kparts;
  if (blocks == 0 || kblocks == 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  sf_prepare_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(ja, jb, kblocks, ksteps, kparts);
  return cudaGetLastError();
}

cudaError_t launch_sf_prepare(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint8_t* img,
                              cudaStream_t stream) {
  return launch_sf_prepare_pair(sf, rows, tile_rows, img, nullptr, 0, 128, nullptr, K, stream);
}

}  // namespace tcg
