// Block-scaled MXFP8 GEMM variants (kind::mxf8f6f4.block_scale.scale_vec::1X,
// E4M3 operands, one e8m0 scale per 32 K elements) and the scale-factor
// rearrangement kernel.
//
// Both variants use N = 256 tiles: a block-scaled MMA issue costs about the
// same time for N = 128 ... 256, so narrower tiles lose in proportion.  TMEM
// (128 lanes x 512 columns, "tcgen05.cp" page, "TMEM shape and replicas")
// then holds one 256-column accumulator and one 16-column scale slot per ring
// stage; the epilogue releases the accumulator as soon as it has read it.
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {


KernelInfo kinfo_mxf8(int cta_group) {
  if (cta_group == 2) {
    using C = GemmCfg<2, 256, 1, 6, KIND_MXF8>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 256, 1, 6, KIND_MXF8>), C::SMEM_BYTES, 2, 256,
            KIND_MXF8, C::THREADS};
  }
  using C = GemmCfg<1, 256, 1, 4, KIND_MXF8>;
  return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 1, 4, KIND_MXF8>), C::SMEM_BYTES, 1, 256,
          KIND_MXF8, C::THREADS};
}

// Packed FP4 (kind::mxf4 with e8m0 scales per 32, kind::mxf4nvf4 with
// unsigned E4M3 scales per 16): a stage carries 256 K of two-per-byte values
// and 8 or 16 scales per row (2 or 4 chunks), so five stages fit for CTA
// pairs (three for single NVFP4 CTAs, whose 256-row B tile is twice as large)
// and four for the 256 x 384 pair tiles (192 B rows per CTA).
KernelInfo kinfo_fp4(int cta_group, bool nvf4, bool wide) {
  if (cta_group == 2 && wide && nvf4) {
    using C = GemmCfg<2, 384, 1, 4, KIND_NVF4>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 384, 1, 4, KIND_NVF4>), C::SMEM_BYTES, 2, 384, KIND_NVF4,
            C::THREADS};
  }
  if (cta_group == 2 && wide) {
    using C = GemmCfg<2, 384, 1, 4, KIND_MXF4>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 384, 1, 4, KIND_MXF4>), C::SMEM_BYTES, 2, 384, KIND_MXF4,
            C::THREADS};
  }
  if (cta_group == 2 && nvf4) {
    using C = GemmCfg<2, 256, 1, 5, KIND_NVF4>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 256, 1, 5, KIND_NVF4>), C::SMEM_BYTES, 2, 256, KIND_NVF4,
            C::THREADS};
  }
  if (cta_group == 2) {
    using C = GemmCfg<2, 256, 1, 5, KIND_MXF4>;
    return {reinterpret_cast<const void*>(&gemm_kernel<2, 256, 1, 5, KIND_MXF4>), C::SMEM_BYTES, 2, 256, KIND_MXF4,
            C::THREADS};
  }
  if (nvf4) {
    using C = GemmCfg<1, 256, 1, 3, KIND_NVF4>;
    return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 1, 3, KIND_NVF4>), C::SMEM_BYTES, 1, 256, KIND_NVF4,
            C::THREADS};
  }
  using C = GemmCfg<1, 256, 1, 4, KIND_MXF4>;
  return {reinterpret_cast<const void*>(&gemm_kernel<1, 256, 1, 4, KIND_MXF4>), C::SMEM_BYTES, 1, 256, KIND_MXF4,
          C::THREADS};
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
// One warp per (128-row chunk of one matrix, group of four K steps); SFA and
// SFB go in the same launch.  The four scale bytes of one row and K step are
// one 32-bit word of the plain layout, and output words 4i..4i+3 of a chunk
// are rows i, 32+i, 64+i, 96+i of the same K step, so lane i reads 16 bytes
// (four K steps) of each of its four rows and writes one 16-byte quad per K
// step: every warp store is 512 contiguous bytes.  Narrower loads and stores
// serve row strides or bases that are not 16-byte multiples.
struct SfJob {
  const uint8_t* sf;
  int64_t rows;
  int64_t tiles;
  int tile_rows;
  int chunks;
  uint32_t* img;
};

constexpr int SF_WARPS = 8;  // warps per block

// kblocks: scale blocks per row of the plain arrays; ksteps: K steps (of
// four blocks) that hold any of them; ksteps_img: K steps of the image, a
// multiple of kch, the K steps per ring stage (1 for MXFP8, 2 for MXFP4, 4
// for NVFP4); the image is [stage][tile][K step of the stage][chunk][512 B].
// Blocks and rows that do not exist hold `fill` (a scale of one in the
// scale's own encoding: the matching operand values are zero, and 0 x NaN
// would not be).
__global__ void __launch_bounds__(32 * SF_WARPS) sf_prepare_kernel(SfJob ja, SfJob jb, int64_t kblocks,
                                                                   int64_t ksteps, int64_t ksteps_img, int kch,
                                                                   uint32_t fill, int64_t kgroups) {
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * SF_WARPS + (threadIdx.x >> 5);
  const int i = threadIdx.x & 31;
  int64_t blk = gw / kgroups;
  const int64_t kg = gw % kgroups;
  const int64_t na = ja.tiles * ja.chunks;
  if (blk >= na + jb.tiles * jb.chunks) return;
  const SfJob j = blk < na ? ja : jb;
  if (blk >= na) blk -= na;
  const int64_t t = blk / j.chunks;
  const int c = static_cast<int>(blk % j.chunks);
  const int64_t row0 = t * j.tile_rows + 128 * c;
  const int valid = static_cast<int>(
      max(static_cast<int64_t>(0), min(min(static_cast<int64_t>(j.tile_rows) - 128 * c, j.rows - row0),
                                       static_cast<int64_t>(128))));
  const int64_t ks0 = 4 * kg;
  // K steps read from the plain arrays (nks) and written to the image (nks_img)
  const int nks = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(4), ksteps - ks0)));
  const int nks_img = static_cast<int>(min(static_cast<int64_t>(4), ksteps_img - ks0));
  const uintptr_t base = reinterpret_cast<uintptr_t>(j.sf);
  const bool quad_loads = nks == 4 && kblocks % 16 == 0 && base % 16 == 0;
  const bool word_loads = kblocks % 4 == 0 && base % 4 == 0;
  uint32_t v[4][4];  // [row group g][K step]
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int rl = 32 * g + i;
    const uint8_t* src = j.sf + (row0 + rl) * kblocks + 4 * ks0;
    if (rl >= valid) {
#pragma unroll
      for (int k = 0; k < 4; ++k) v[g][k] = fill;
    } else if (quad_loads) {
      const uint4 q = *reinterpret_cast<const uint4*>(src);
      v[g][0] = q.x;
      v[g][1] = q.y;
      v[g][2] = q.z;
      v[g][3] = q.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (k >= nks) {
          v[g][k] = fill;
        } else if (word_loads) {
          v[g][k] = reinterpret_cast<const uint32_t*>(src)[k];
        } else {
          uint32_t w = 0u;
          for (int b = 0; b < 4; ++b) {
            const int64_t kb = 4 * (ks0 + k) + b;
            w |= (kb < kblocks ? static_cast<uint32_t>(src[4 * k + b]) : (fill & 0xFFu)) << (8 * b);
          }
          v[g][k] = w;
        }
      }
    }
  }
  const bool quad_stores = reinterpret_cast<uintptr_t>(j.img) % 16 == 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k < nks_img) {
      const int64_t ks = ks0 + k;
      uint32_t* dst = j.img + ((((ks / kch) * j.tiles + t) * kch + ks % kch) * j.chunks + c) * 128 + 4 * i;
      if (quad_stores) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(v[0][k], v[1][k], v[2][k], v[3][k]);
      } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) dst[g] = v[g][k];
      }
    }
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

ScaleFormat scale_format(tcg_input t) {
  // MXFP8 / FP6 / FP4 on kind::mxf8f6f4: e8m0 per 32, one 128-K step per stage;
  // packed MXFP4: e8m0 per 32, stages of 256 K; NVFP4: unsigned E4M3 per 16,
  // stages of 256 K
  if (t == TCG_IN_E2M1) return {32, 2, 0x7Fu};
  if (t == TCG_IN_NVF4) return {16, 4, 0x38u};
  return {32, 1, 0x7Fu};
}

int64_t sf_image_bytes_fmt(tcg_input t, int64_t rows, int64_t K, int tile_rows) {
  const ScaleFormat f = scale_format(t);
  const int64_t kblocks = (K + f.block - 1) / f.block;
  const int64_t ksteps = (kblocks + 3) / 4;
  const int64_t ksteps_img = (ksteps + f.kch - 1) / f.kch * f.kch;
  return ksteps_img * ((rows + tile_rows - 1) / tile_rows) * ((tile_rows + 127) / 128) * 512;
}

cudaError_t launch_sf_prepare_pair(tcg_input t, const uint8_t* sfa, int64_t rows_a, int tile_a, uint8_t* img_a,
                                   const uint8_t* sfb, int64_t rows_b, int tile_b, uint8_t* img_b, int64_t K,
                                   cudaStream_t stream) {
  const ScaleFormat f = scale_format(t);
  const int64_t kblocks = (K + f.block - 1) / f.block;
  const int64_t ksteps = (kblocks + 3) / 4;
  const int64_t ksteps_img = (ksteps + f.kch - 1) / f.kch * f.kch;
  const int64_t kgroups = (ksteps_img + 3) / 4;
  const SfJob ja = make_job(sfa, rows_a, tile_a, img_a);
  const SfJob jb = make_job(sfb, rows_b, tile_b, img_b);
  const int64_t warps = (ja.tiles * ja.chunks + jb.tiles * jb.chunks) * kgroups;
  if (warps == 0 || kblocks == 0) return cudaSuccess;
  const int64_t blocks = (warps + SF_WARPS - 1) / SF_WARPS;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  const uint32_t fill4 = f.fill * 0x01010101u;
  sf_prepare_kernel<<<static_cast<unsigned>(blocks), 32 * SF_WARPS, 0, stream>>>(ja, jb, kblocks, ksteps, ksteps_img,
                                                                                f.kch, fill4, kgroups);
  return cudaGetLastError();
}

cudaError_t launch_sf_prepare(tcg_input t, const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint8_t* img,
                              cudaStream_t stream) {
  return launch_sf_prepare_pair(t, sf, rows, tile_rows, img, nullptr, 0, 128, nullptr, K, stream);
}

}  // namespace tcg
