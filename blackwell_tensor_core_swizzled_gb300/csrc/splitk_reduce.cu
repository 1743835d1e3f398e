// Final step of split-K / stream-K GEMMs: every output tile computed in parts
// has one fp32 partial per contributing unit in the workspace slots (written
// by the GEMM kernel's epilogue); this kernel sums them in K order and writes
// D (or, for a transposed product, D's transpose).  One thread per (tile, CTA
// of a pair, row, 4 columns): 16-byte slot loads (all slots of a thread are
// independent, so they overlap), an fp32 sum, the output conversion and the
// stores.  Tiles computed whole by one unit were stored to D directly and are
// skipped.  Launched as a programmatic dependent of the GEMM (its launch
// overlaps the GEMM's last CTAs); it waits for the GEMM's completion and
// memory flush before reading the slots.
#include "common.h"
#include "gemm_kernel.cuh"

namespace tcg {

__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ GemmParams p, int cg,
                                                            int num_clusters) {
  griddep_wait();
  const int q4 = p.bn / 4;
  const int64_t per_rank = static_cast<int64_t>(p.w_rows) * q4;
  const int64_t per_tile = cg * per_rank;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int tile = static_cast<int>(idx / per_tile);
  if (tile >= p.num_tiles) return;
  int64_t r = idx - tile * per_tile;
  const int rank = static_cast<int>(r / per_rank);
  r -= rank * per_rank;
  // rows fastest for a transposed D (a warp's 32 rows are one contiguous run
  // of each D row), else 4-column groups fastest
  int lrow, c4;
  if (p.d_trans) {
    c4 = static_cast<int>(r / p.w_rows);
    lrow = static_cast<int>(r - static_cast<int64_t>(c4) * p.w_rows);
  } else {
    lrow = static_cast<int>(r / q4);
    c4 = static_cast<int>(r - static_cast<int64_t>(lrow) * q4);
  }
  // contributing units: `split` consecutive slots, or under stream-K the
  // clusters c0 .. c0+n-1 whose ranges meet the tile; cluster c's slot is
  // 2c for its head (its range starts inside this tile) else 2c+1 (start(c)
  // = floor(c*T/G) < s0 exactly when c*T < s0*G)
  int n = p.split;
  int64_t c0 = 0, T = 0, s0g = 0;
  if (p.stream_k) {
    T = static_cast<int64_t>(p.num_tiles) * p.num_k_blocks;
    const int64_t s0 = static_cast<int64_t>(tile) * p.num_k_blocks;
    const int64_t G = num_clusters;
    c0 = ((s0 + 1) * G - 1) / T;
    n = static_cast<int>(((s0 + p.num_k_blocks) * G - 1) / T - c0 + 1);
    s0g = s0 * G;
    if (n == 1) return;  // computed whole, stored directly
  }
  int mt, nt;
  tile_coords(tile, p, mt, nt);
  const int64_t row = static_cast<int64_t>(mt) * 128 * cg + 128 * rank + lrow;
  const int col = nt * p.bn + 4 * c4;
  if (row >= p.M || col >= p.N) return;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int j = 0; j < n; ++j) {
    int64_t slot;
    if (p.stream_k) {
      const int64_t cc = c0 + j;
      slot = 2 * cc + (cc * T < s0g ? 1 : 0);
    } else {
      slot = static_cast<int64_t>(tile) * p.split + j;
    }
    const int64_t z = slot * cg + rank;
    const float4 t = __ldcg(reinterpret_cast<const float4*>(p.w + (z * p.w_rows + lrow) * p.bn + 4 * c4));
    v.x += t.x;
    v.y += t.y;
    v.z += t.z;
    v.w += t.w;
  }
  const bool full4 = col + 3 < p.N;
  const float vals[4] = {v.x, v.y, v.z, v.w};
  if (p.d_trans) {
    // element (row, col + e) of the transposed product is D[(col + e) * ldd + row]
    for (int e = 0; e < 4; ++e) {
      if (col + e >= p.N) break;
      const int64_t off = static_cast<int64_t>(col + e) * p.ldd + row;
      if (p.d_type == OUT_F32)
        reinterpret_cast<float*>(p.D)[off] = vals[e];
      else if (p.d_type == OUT_BF16)
        reinterpret_cast<uint16_t*>(p.D)[off] = __bfloat16_as_ushort(__float2bfloat16_rn(vals[e]));
      else
        reinterpret_cast<uint16_t*>(p.D)[off] = __half_as_ushort(__float2half_rn(vals[e]));
    }
    return;
  }
  if (p.d_type == OUT_F32) {
    float* dst = reinterpret_cast<float*>(p.D) + row * p.ldd + col;
    if (full4 && p.d_vec_ok) {
      *reinterpret_cast<float4*>(dst) = v;
    } else {
      for (int e = 0; e < 4; ++e)
        if (col + e < p.N) dst[e] = vals[e];
    }
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.D) + row * p.ldd + col;
    const bool bf = p.d_type == OUT_BF16;
    const uint32_t lo = bf ? pack_bf16(__float_as_uint(vals[0]), __float_as_uint(vals[1]))
                           : pack_f16(__float_as_uint(vals[0]), __float_as_uint(vals[1]));
    const uint32_t hi = bf ? pack_bf16(__float_as_uint(vals[2]), __float_as_uint(vals[3]))
                           : pack_f16(__float_as_uint(vals[2]), __float_as_uint(vals[3]));
    if (full4 && p.d_vec_ok) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    } else {
      const uint32_t w2[2] = {lo, hi};
      for (int e = 0; e < 4; ++e)
        if (col + e < p.N) dst[e] = static_cast<uint16_t>((w2[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
    }
  }
}

cudaError_t launch_splitk_reduce(const GemmParams& p, int cg, int num_clusters, cudaStream_t stream) {
  const int64_t threads = static_cast<int64_t>(p.num_tiles) * cg * p.w_rows * (p.bn / 4);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, p, cg, num_clusters);
}

}  // namespace tcg
