// Single-CTA layout probes.  Each exposes one mechanism the tcgen05 / ldmatrix
// documentation pages describe, so the tests can compare it bit for bit with
// those pages' layout rules:
//   * TMEM st/ld round trip ("tcgen05.ld / tcgen05.st" page, Layout B example;
//     the copy_async -> tcgen05_ldst page's 128x8 demonstration);
//   * tcgen05.cp from a descriptor-walked shared image ("tcgen05.cp" page,
//     shape table and "Shared descriptor address walk"), plain or with the
//     FP4 / FP6 decompression ("Native FP4/FP6 decompression");
//   * tcgen05.ld register images of the 16-row shapes ("Native images");
//   * one MMA tile with generic-store swizzled operands ("tcgen05.mma" page,
//     "four K16 issues" example), dense or with the weight-stationary .ws
//     opcode ("Weight-stationary and block scaling");
//   * one MMA tile whose A operand is in tensor memory (Layout D, M = 128);
//   * a weight-stationary M = 64 tile, A from shared memory or from a
//     two-bank TMEM image, returning the raw accumulator image;
//   * MMAs reading operand images the caller laid out, through descriptors
//     the caller chose (K-major or MN-major, swizzle modes 0..4): the
//     hardware's descriptor walk against a layout model ("tcgen05.mma" page,
//     "Shared descriptors are byte-stride contracts", "swizzle=4");
//   * ldmatrix .x2 into separated register slots ("ldmatrix / stmatrix" page
//     example) and stmatrix .x1/.x2/.x4 with and without .trans ("Transpose
//     and stores");
//   * tcgen05.ld / st .16x32bx2 split accesses ("tcgen05.ld / tcgen05.st"
//     page, "Split accesses: 16x32bx2");
//   * a bounded wait that runs out (failure detection without a GPU fault).
#include <cuda_runtime.h>

#include "common.h"
#include "gemm_kernel.cuh"
#include "tmem_ldst.cuh"

namespace tcg {
namespace {

__device__ __forceinline__ WaitCtx probe_wait_ctx(unsigned long long* err, uint64_t timeout_ns,
                                                  volatile uint32_t* abort_flag) {
  return WaitCtx{timeout_ns, err, abort_flag};
}

// ------------------------------------------------------------------ TMEM round trip

template <int NC>
__device__ __forceinline__ void st_x(uint32_t taddr, const uint32_t* r) {
  if constexpr (NC == 1) stx_32x32b_x1(taddr, r);
  if constexpr (NC == 2) stx_32x32b_x2(taddr, r);
  if constexpr (NC == 4) stx_32x32b_x4(taddr, r);
  if constexpr (NC == 8) stx_32x32b_x8(taddr, r);
  if constexpr (NC == 16) stx_32x32b_x16(taddr, r);
  if constexpr (NC == 32) stx_32x32b_x32(taddr, r);
  if constexpr (NC == 64) stx_32x32b_x64(taddr, r);
}

template <int NC>
__device__ __forceinline__ void ld_x(uint32_t taddr, uint32_t* r) {
  if constexpr (NC == 1) ldx_32x32b_x1(taddr, r);
  if constexpr (NC == 2) ldx_32x32b_x2(taddr, r);
  if constexpr (NC == 4) ldx_32x32b_x4(taddr, r);
  if constexpr (NC == 8) ldx_32x32b_x8(taddr, r);
  if constexpr (NC == 16) ldx_32x32b_x16(taddr, r);
  if constexpr (NC == 32) ldx_32x32b_x32(taddr, r);
  if constexpr (NC == 64) ldx_32x32b_x64(taddr, r);
}

template <int NC>
__global__ void __launch_bounds__(128, 1) probe_tmem_roundtrip_kernel(const uint32_t* in, uint32_t* out) {
  constexpr uint32_t COLS = NC < 32 ? 32 : NC;
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), COLS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = slot + (static_cast<uint32_t>(32 * warp) << 16);
  uint32_t r[NC];
#pragma unroll
  for (int j = 0; j < NC; ++j) r[j] = in[t * NC + j];
  st_x<NC>(taddr, r);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t o[NC];
  ld_x<NC>(taddr, o);
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < NC; ++j) out[t * NC + j] = o[j];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, COLS);
}

// ------------------------------------------------------------------ tcgen05.cp

constexpr int CP_IMAGE_MAX_WORDS = 12288;  // 48 KiB

__global__ void __launch_bounds__(128, 1) probe_cp_kernel(const uint32_t* image, int image_words, int shape,
                                                          uint32_t origin, uint64_t desc_hi, uint32_t* out,
                                                          unsigned long long* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t* img = reinterpret_cast<uint32_t*>(smem_raw + (base - raw));
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < image_words; i += blockDim.x) img[i] = image[i];
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), 32);
    tmem_relinquish<1>();
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Fill the 8 columns with a sentinel so cells the copy does not write show.
  const uint32_t taddr = slot + (static_cast<uint32_t>(32 * warp) << 16);
  uint32_t sent[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) sent[j] = 0xDEADBEEFu;
  stx_32x32b_x8(taddr, sent);
  tc_wait_st();
  fence_proxy_async_shared();  // generic-proxy image writes -> async proxy (tcgen05.cp)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint64_t d = sdesc(base + origin, desc_hi);
    // shape + 4 * format: format 1 / 2 expand packed FP4 / FP6 blocks
    // ("tcgen05.cp" page, "Native FP4/FP6 decompression")
    switch (shape) {
      case 0: asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(slot), "l"(d) : "memory"); break;
      case 1: asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(slot), "l"(d) : "memory"); break;
      case 2: asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(slot), "l"(d) : "memory"); break;
      case 3: asm volatile("tcgen05.cp.cta_group::1.4x256b [%0], %1;" ::"r"(slot), "l"(d) : "memory"); break;
      case 4:
        asm volatile("tcgen05.cp.cta_group::1.128x256b.b8x16.b4x16_p64 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
      case 5:
        asm volatile("tcgen05.cp.cta_group::1.128x128b.b8x16.b4x16_p64 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
      case 6:
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4.b8x16.b4x16_p64 [%0], %1;" ::"r"(slot), "l"(d)
                     : "memory");
        break;
      case 7:
        asm volatile("tcgen05.cp.cta_group::1.4x256b.b8x16.b4x16_p64 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
      case 8:
        asm volatile("tcgen05.cp.cta_group::1.128x256b.b8x16.b6x16_p32 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
      case 9:
        asm volatile("tcgen05.cp.cta_group::1.128x128b.b8x16.b6x16_p32 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
      case 10:
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4.b8x16.b6x16_p32 [%0], %1;" ::"r"(slot), "l"(d)
                     : "memory");
        break;
      default:
        asm volatile("tcgen05.cp.cta_group::1.4x256b.b8x16.b6x16_p32 [%0], %1;" ::"r"(slot), "l"(d) : "memory");
        break;
    }
    tc_commit<1>(smem_u32(&bar));
  }
  const bool ok = warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
  tc_fence_after();
  uint32_t o[8];
  ldx_32x32b_x8(taddr, o);
  tc_wait_ld();
  if (ok) {
#pragma unroll
    for (int j = 0; j < 8; ++j) out[threadIdx.x * 8 + j] = o[j];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, 32);
}

// ------------------------------------------------------------------ ld shapes

template <int SHAPE, int NUM>
__device__ __forceinline__ void ld_shape(uint32_t taddr, uint32_t* r) {
  if constexpr (SHAPE == 0) {
    if constexpr (NUM == 1) ldx_32x32b_x1(taddr, r);
    if constexpr (NUM == 2) ldx_32x32b_x2(taddr, r);
    if constexpr (NUM == 4) ldx_32x32b_x4(taddr, r);
    if constexpr (NUM == 8) ldx_32x32b_x8(taddr, r);
    if constexpr (NUM == 16) ldx_32x32b_x16(taddr, r);
    if constexpr (NUM == 32) ldx_32x32b_x32(taddr, r);
  } else if constexpr (SHAPE == 1) {
    if constexpr (NUM == 1) ldx_16x64b_x1(taddr, r);
    if constexpr (NUM == 2) ldx_16x64b_x2(taddr, r);
    if constexpr (NUM == 4) ldx_16x64b_x4(taddr, r);
    if constexpr (NUM == 8) ldx_16x64b_x8(taddr, r);
    if constexpr (NUM == 16) ldx_16x64b_x16(taddr, r);
  } else if constexpr (SHAPE == 2) {
    if constexpr (NUM == 1) ldx_16x128b_x1(taddr, r);
    if constexpr (NUM == 2) ldx_16x128b_x2(taddr, r);
    if constexpr (NUM == 4) ldx_16x128b_x4(taddr, r);
    if constexpr (NUM == 8) ldx_16x128b_x8(taddr, r);
  } else {
    if constexpr (NUM == 1) ldx_16x256b_x1(taddr, r);
    if constexpr (NUM == 2) ldx_16x256b_x2(taddr, r);
    if constexpr (NUM == 4) ldx_16x256b_x4(taddr, r);
  }
}

template <int SHAPE, int NUM>
__global__ void __launch_bounds__(128, 1) probe_ld_shape_kernel(const uint32_t* in, int half, uint32_t* out) {
  constexpr int REGS = SHAPE == 0 ? NUM : SHAPE == 1 ? NUM : SHAPE == 2 ? 2 * NUM : 4 * NUM;
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), 32);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t lane_base = slot + (static_cast<uint32_t>(32 * warp) << 16);
  uint32_t img[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) img[j] = in[t * 32 + j];
  stx_32x32b_x32(lane_base, img);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t taddr = lane_base + (SHAPE == 0 ? 0u : (static_cast<uint32_t>(16 * half) << 16));
  uint32_t r[REGS];
  ld_shape<SHAPE, NUM>(taddr, r);
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < REGS; ++j) out[t * REGS + j] = r[j];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, 32);
}

// ------------------------------------------------------------------ one MMA tile

// A (128 x K) and B (N x K), both K-major 16-bit, written with ordinary
// stores into 128B-swizzled shared tiles (descriptor (LDO 16, SDO 1024,
// swizzle 128B): row r at (r/8)*1024 + (r%8)*128, element k at 2k, then the
// mode-3 XOR), K/16 MMA issues whose start address advances 32 bytes each.
__global__ void __launch_bounds__(128, 1) probe_mma_tile_kernel(const uint16_t* A, const uint16_t* B, int N, int K,
                                                                uint32_t idesc, int ws, float* D,
                                                                unsigned long long* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  const uint32_t a_base = base;               // 128 rows x 128 B
  const uint32_t b_base = base + 128 * 128;   // up to 256 rows x 128 B
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  // zero both tiles, then scatter the operands at their swizzled addresses
  for (int i = t; i < (128 + 256) * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(g)[i] = 0u;
  __syncthreads();
  for (int i = t; i < 128 * K; i += blockDim.x) {
    const int m = i / K, k = i % K;
    const uint32_t logical = a_base + (m / 8) * 1024u + (m % 8) * 128u + 2u * k;
    *reinterpret_cast<uint16_t*>(g + (swizzle_addr(logical, SW_128B) - base)) = A[i];
  }
  for (int i = t; i < N * K; i += blockDim.x) {
    const int n = i / K, k = i % K;
    const uint32_t logical = b_base + (n / 8) * 1024u + (n % 8) * 128u + 2u * k;
    *reinterpret_cast<uint16_t*>(g + (swizzle_addr(logical, SW_128B) - base)) = B[i];
  }
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(N)) ncols <<= 1;
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), ncols);
    tmem_relinquish<1>();
  }
  if (t == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t == 0) {
    const uint64_t hi = sdesc_hi(16, 1024, SW_128B);
    for (int kr = 0; kr < K / 16; ++kr) {
      const uint64_t ad = sdesc(a_base + 32u * kr, hi), bd = sdesc(b_base + 32u * kr, hi);
      if (ws) {
        // weight-stationary opcode ("tcgen05.mma" page, "Weight-stationary and
        // block scaling": selected in the opcode; M128 .ws uses Layout D)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.ws.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(slot),
            "l"(ad), "l"(bd), "r"(idesc), "r"(kr > 0 ? 1u : 0u)
            : "memory");
      } else {
        mma_f16<1>(slot, ad, bd, idesc, kr > 0);
      }
    }
    tc_commit<1>(smem_u32(&bar));
  }
  const bool ok = warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
  tc_fence_after();
  const uint32_t tb = slot + (static_cast<uint32_t>(32 * warp) << 16);
  for (int c = 0; c < N; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tb + c, r);
    tc_wait_ld();
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c + j < N) D[t * N + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, ncols);
}

// ------------------------------------------------------------------ A operand in TMEM

// One MMA tile whose A operand sits in tensor memory ("tcgen05.mma" page,
// "Operands and repeat axes": A from shared memory or TMEM, "A in TMEM is
// packed according to its input format"; M = 128 uses Layout D): thread t
// writes row t of A (K 16-bit values, two per 32-bit column, the lower K in
// the low half) to TMEM lane t at columns [A_COL, A_COL + K/2) with
// tcgen05.st .32x32b; B (N x K, K-major) is written into a 128B-swizzled
// shared tile as in probe_mma_tile; K/16 MMAs read A from column A_COL + 8j
// and B through descriptors advancing 32 bytes; D drains with .32x32b.
constexpr uint32_t TMEM_A_COL = 256;

__global__ void __launch_bounds__(128, 1) probe_mma_tmem_a_kernel(const uint16_t* A, const uint16_t* B, int N, int K,
                                                                  uint32_t idesc, float* D, unsigned long long* err,
                                                                  uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  for (int i = t; i < 256 * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(g)[i] = 0u;
  __syncthreads();
  for (int i = t; i < N * K; i += blockDim.x) {
    const int n = i / K, k = i % K;
    const uint32_t logical = base + (n / 8) * 1024u + (n % 8) * 128u + 2u * k;
    *reinterpret_cast<uint16_t*>(g + (swizzle_addr(logical, SW_128B) - base)) = B[i];
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), 512);
    tmem_relinquish<1>();
  }
  if (t == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // row t of A into lane t: 32 columns hold K <= 64 values
  uint32_t words[32];
#pragma unroll
  for (int c = 0; c < 32; ++c)
    words[c] = 2 * c < K ? (static_cast<uint32_t>(A[t * K + 2 * c]) | (static_cast<uint32_t>(A[t * K + 2 * c + 1]) << 16))
                         : 0u;
  const uint32_t lane_base = slot + (static_cast<uint32_t>(32 * warp) << 16);
  stx_32x32b_x32(lane_base + TMEM_A_COL, words);
  tc_wait_st();
  fence_proxy_async_shared();  // B's generic stores -> the MMA's async reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t == 0) {
    const uint64_t hi = sdesc_hi(16, 1024, SW_128B);
    for (int kr = 0; kr < K / 16; ++kr)
      mma_f16_tmem_a(slot, slot + TMEM_A_COL + 8u * kr, sdesc(base + 32u * kr, hi), idesc, kr > 0);
    tc_commit<1>(smem_u32(&bar));
  }
  const bool ok = warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
  tc_fence_after();
  for (int c = 0; c < N; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(lane_base + c, r);
    tc_wait_ld();
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c + j < N) D[t * N + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, 512);
}

// ------------------------------------------------------------------ weight-stationary M = 64

// One weight-stationary MMA tile of M = 64 ("tcgen05.mma" page,
// "Weight-stationary and block scaling": M64 .ws, N = 64 / 128 / 256, CTA
// group 1; with A in TMEM "an atom bank axis: A ends in (2,64,K)").  A comes
// from a 128B-swizzled shared tile (64 rows x K) or, with a_tmem, from tensor
// memory: thread t writes row t of the (2, 64, K) bank image -- bank t / 64,
// row t % 64 -- to lane t at columns [TMEM_A_COL, TMEM_A_COL + K/2).  B (N x
// K, K-major) as in probe_mma_tile.  The raw accumulator image, 128 lanes x
// N/2 columns, is read back with .32x32b and returned lane-major, so the test
// can compare it with a layout model.
__global__ void __launch_bounds__(128, 1) probe_mma_ws64_kernel(const uint16_t* A, const uint16_t* B, int N, int K,
                                                                int a_tmem, uint32_t idesc, uint32_t* out,
                                                                unsigned long long* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* g = smem_raw + (base - raw);
  const uint32_t a_base = base;              // 64 rows x 128 B (and zero rows after)
  const uint32_t b_base = base + 128 * 128;  // up to 256 rows x 128 B
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  for (int i = t; i < (128 + 256) * 128 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(g)[i] = 0u;
  __syncthreads();
  if (!a_tmem) {
    for (int i = t; i < 64 * K; i += blockDim.x) {
      const int m = i / K, k = i % K;
      const uint32_t logical = a_base + (m / 8) * 1024u + (m % 8) * 128u + 2u * k;
      *reinterpret_cast<uint16_t*>(g + (swizzle_addr(logical, SW_128B) - base)) = A[i];
    }
  }
  for (int i = t; i < N * K; i += blockDim.x) {
    const int n = i / K, k = i % K;
    const uint32_t logical = b_base + (n / 8) * 1024u + (n % 8) * 128u + 2u * k;
    *reinterpret_cast<uint16_t*>(g + (swizzle_addr(logical, SW_128B) - base)) = B[i];
  }
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), 512);
    tmem_relinquish<1>();
  }
  if (t == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t lane_base = slot + (static_cast<uint32_t>(32 * warp) << 16);
  if (a_tmem) {
    uint32_t words[32];
#pragma unroll
    for (int c = 0; c < 32; ++c)
      words[c] = 2 * c < K
                     ? (static_cast<uint32_t>(A[t * K + 2 * c]) | (static_cast<uint32_t>(A[t * K + 2 * c + 1]) << 16))
                     : 0u;
    stx_32x32b_x32(lane_base + TMEM_A_COL, words);
    tc_wait_st();
  }
  fence_proxy_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t == 0) {
    const uint64_t hi = sdesc_hi(16, 1024, SW_128B);
    for (int kr = 0; kr < K / 16; ++kr) {
      const uint64_t bd = sdesc(b_base + 32u * kr, hi);
      if (a_tmem)
        mma_ws_f16_tmem_a(slot, slot + TMEM_A_COL + 8u * kr, bd, idesc, kr > 0);
      else
        mma_ws_f16(slot, sdesc(a_base + 32u * kr, hi), bd, idesc, kr > 0);
    }
    tc_commit<1>(smem_u32(&bar));
  }
  const bool ok = warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
  tc_fence_after();
  const int cols = N / 2;
  for (int c = 0; c < cols; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(lane_base + c, r);
    tc_wait_ld();
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c + j < cols) out[t * cols + c + j] = r[j];
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, 512);
}

// ------------------------------------------------------------------ MMA from caller images

// One operand of tcg_probe_mma_image as the kernel sees it: where its image
// sits in the CTA's shared memory and the descriptor of each issue.
struct ImageOperand {
  const uint4* image;
  int words16;        // image size in 16-byte units
  uint64_t desc_hi;   // LDO, SDO, version, layout type
  uint32_t start[8];  // descriptor origin of issue j, bytes from the region start
};

constexpr uint32_t MMA_IMAGE_REGION = 96u * 1024u;  // bytes per operand region

// A's region at the 1024-byte aligned base, B's MMA_IMAGE_REGION later; both
// regions are zeroed, the images copied in with ordinary stores, and thread 0
// issues `ksteps` MMAs of one kind (kind::f16 for f16 / bf16, kind::tf32),
// accumulation off on the first.  The device computes no layout: which
// element each descriptor step reads is decided by the images alone.
__global__ void __launch_bounds__(128, 1) probe_mma_image_kernel(ImageOperand a, ImageOperand b, int tf32,
                                                                 uint32_t idesc, int N, int ksteps, float* D,
                                                                 unsigned long long* err, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t slot;
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint4* g = reinterpret_cast<uint4*>(smem_raw + (base - raw));
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  constexpr int REGION16 = MMA_IMAGE_REGION / 16;
  for (int i = t; i < 2 * REGION16; i += blockDim.x) g[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  for (int i = t; i < a.words16; i += blockDim.x) g[i] = a.image[i];
  for (int i = t; i < b.words16; i += blockDim.x) g[REGION16 + i] = b.image[i];
  uint32_t ncols = 32;
  while (ncols < static_cast<uint32_t>(N)) ncols <<= 1;
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), ncols);
    tmem_relinquish<1>();
  }
  if (t == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  fence_proxy_async_shared();  // generic-proxy image stores -> the MMA's async reads
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (t == 0) {
    for (int j = 0; j < ksteps; ++j) {
      const uint64_t ad = sdesc(base + a.start[j], a.desc_hi);
      const uint64_t bd = sdesc(base + MMA_IMAGE_REGION + b.start[j], b.desc_hi);
      if (tf32)
        mma_tf32<1>(slot, ad, bd, idesc, j > 0);
      else
        mma_f16<1>(slot, ad, bd, idesc, j > 0);
    }
    tc_commit<1>(smem_u32(&bar));
  }
  const bool ok = warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
  tc_fence_after();
  const uint32_t tb = slot + (static_cast<uint32_t>(32 * warp) << 16);
  for (int c = 0; c < N; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(tb + c, r);
    tc_wait_ld();
    if (ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c + j < N) D[t * N + c + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, ncols);
}

// ------------------------------------------------------------------ split accesses 16x32bx2

// Every thread stores in[t*32 .. t*32+32) to TMEM lane t, columns [0, 32),
// and zeroes columns [32, 64); each warp then loads its quadrant with
// tcgen05.ld .16x32bx2.x<NUM> (second access IMM after the first) into
// out_ld, stores distinct words 0x10000 * t + r + 1 with tcgen05.st
// .16x32bx2.x<NUM> at column 32, and every thread reads columns [32, 64) of
// its lane back into out_st.
template <int NUM, uint32_t IMM>
__global__ void __launch_bounds__(128, 1) probe_split_kernel(const uint32_t* in, uint32_t* out_ld, uint32_t* out_st) {
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  if (warp == 0) {
    tmem_alloc<1>(smem_u32(&slot), 64);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t lane_base = slot + (static_cast<uint32_t>(32 * warp) << 16);
  uint32_t img[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) img[j] = in[t * 32 + j];
  stx_32x32b_x32(lane_base, img);
#pragma unroll
  for (int j = 0; j < 32; ++j) img[j] = 0u;
  stx_32x32b_x32(lane_base + 32, img);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  uint32_t r[NUM];
  if constexpr (NUM == 1) ldx_16x32bx2_x1<IMM>(lane_base, r);
  if constexpr (NUM == 2) ldx_16x32bx2_x2<IMM>(lane_base, r);
  if constexpr (NUM == 4) ldx_16x32bx2_x4<IMM>(lane_base, r);
  if constexpr (NUM == 8) ldx_16x32bx2_x8<IMM>(lane_base, r);
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < NUM; ++j) out_ld[t * NUM + j] = r[j];
#pragma unroll
  for (int j = 0; j < NUM; ++j) r[j] = 0x10000u * static_cast<uint32_t>(t) + static_cast<uint32_t>(j) + 1u;
  if constexpr (NUM == 1) stx_16x32bx2_x1<IMM>(lane_base + 32, r);
  if constexpr (NUM == 2) stx_16x32bx2_x2<IMM>(lane_base + 32, r);
  if constexpr (NUM == 4) stx_16x32bx2_x4<IMM>(lane_base + 32, r);
  if constexpr (NUM == 8) stx_16x32bx2_x8<IMM>(lane_base + 32, r);
  tc_wait_st();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  ldx_32x32b_x32(lane_base + 32, img);
  tc_wait_ld();
#pragma unroll
  for (int j = 0; j < 32; ++j) out_st[t * 32 + j] = img[j];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<1>(slot, 64);
}

// ------------------------------------------------------------------ stmatrix

// One warp: lane l holds COUNT words regs[l*4 .. l*4+COUNT) and provides the
// shared address of row (l % (8*COUNT)) of the matrices: row_off[that row]
// bytes (masked to a 16-byte multiple below 1024) into a zeroed 1 KB buffer; stmatrix .m8n8.x<COUNT>[.trans].b16
// writes, and the buffer comes back in out (256 words).
template <int COUNT, bool TRANS>
__global__ void probe_stmatrix_kernel(const uint32_t* regs, const uint32_t* row_off, uint32_t* out) {
  __shared__ __align__(16) uint32_t sm[256];
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < 256; i += 32) sm[i] = 0u;
  __syncwarp();
  const uint32_t addr = smem_u32(sm) + (row_off[lane % (8 * COUNT)] & 1008u);
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = regs[lane * 4 + i];
  if constexpr (COUNT == 1 && !TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x1.shared.b16 [%0], {%1};" ::"r"(addr), "r"(r[0]) : "memory");
  if constexpr (COUNT == 1 && TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x1.trans.shared.b16 [%0], {%1};" ::"r"(addr), "r"(r[0]) : "memory");
  if constexpr (COUNT == 2 && !TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x2.shared.b16 [%0], {%1, %2};" ::"r"(addr), "r"(r[0]), "r"(r[1])
                 : "memory");
  if constexpr (COUNT == 2 && TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x2.trans.shared.b16 [%0], {%1, %2};" ::"r"(addr), "r"(r[0]), "r"(r[1])
                 : "memory");
  if constexpr (COUNT == 4 && !TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
  if constexpr (COUNT == 4 && TRANS)
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
  __syncwarp();
  for (int i = lane; i < 256; i += 32) out[i] = sm[i];
}

// ------------------------------------------------------------------ ldmatrix

// x (16,4,2) row-major words; shared layout (16,4,2):(8,1,128).  Matrix m,
// row r of issue k is shared row (2r+m, :, k); lane 8m+r provides its address
// (lanes 16..31 repeat lanes 0..15).  The register words of issue k land in
// slots 8k (matrix 0) and 8k+2 (matrix 1).
__global__ void probe_ldmatrix_kernel(const uint32_t* x, uint32_t* out) {
  __shared__ __align__(16) uint32_t sm[256];
  const int lane = threadIdx.x & 31;
  for (int i = lane; i < 256; i += 32) sm[i] = 0u;
  __syncwarp();
  for (int q = 0; q < 4; ++q) {
    const int n = lane + 32 * q;
    const int i = n / 8, j = (n / 2) % 4, k = n % 2;
    sm[8 * i + j + 128 * k] = x[n];
  }
  __syncwarp();
  uint32_t raw[12];
#pragma unroll
  for (int i = 0; i < 12; ++i) raw[i] = 4294966519u;
  const int l = lane & 15;
  const int m = l >> 3, r = l & 7;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t addr = smem_u32(&sm[8 * (2 * r + m) + 128 * k]);
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(raw[8 * k]), "=r"(raw[8 * k + 2])
                 : "r"(addr));
  }
#pragma unroll
  for (int i = 0; i < 12; ++i) out[lane * 12 + i] = raw[i];
}

// ------------------------------------------------------------------ bounded wait

__global__ void probe_wait_timeout_kernel(unsigned long long* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // nobody ever arrives
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  warp_wait(smem_u32(&bar), 0, probe_wait_ctx(err, timeout_ns, &abort_flag), SITE_PROBE);
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int finish_launch(int launches) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda(e);
  set_launch_count(launches);
  return TCG_OK;
}

}  // namespace
}  // namespace tcg

using namespace tcg;

extern "C" int tcg_probe_tmem_roundtrip(const uint32_t* in, uint32_t* out, int ncols, void* stream) {
  if (!in || !out) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaStream_t s = as_stream(stream);
  switch (ncols) {
    case 1: probe_tmem_roundtrip_kernel<1><<<1, 128, 0, s>>>(in, out); break;
    case 2: probe_tmem_roundtrip_kernel<2><<<1, 128, 0, s>>>(in, out); break;
    case 4: probe_tmem_roundtrip_kernel<4><<<1, 128, 0, s>>>(in, out); break;
    case 8: probe_tmem_roundtrip_kernel<8><<<1, 128, 0, s>>>(in, out); break;
    case 16: probe_tmem_roundtrip_kernel<16><<<1, 128, 0, s>>>(in, out); break;
    case 32: probe_tmem_roundtrip_kernel<32><<<1, 128, 0, s>>>(in, out); break;
    case 64: probe_tmem_roundtrip_kernel<64><<<1, 128, 0, s>>>(in, out); break;
    default: return TCG_ERR_INVALID;
  }
  return finish_launch(1);
}

extern "C" int tcg_probe_cp(const uint32_t* image, int image_words, int shape, uint32_t origin_bytes, uint32_t ldo,
                            uint32_t sdo, int swizzle, uint32_t* out, void* stream) {
  if (!image || !out || image_words <= 0 || image_words > CP_IMAGE_MAX_WORDS) return TCG_ERR_INVALID;
  if (shape < 0 || shape > 11 || swizzle < 0 || swizzle > 3) return TCG_ERR_INVALID;
  if (!sdesc_fields_ok(origin_bytes, ldo, sdo, swizzle, 0)) return TCG_ERR_INVALID;
  // The copy's whole walk must stay inside the image, and every row group it
  // touches must be backed whole: the descriptor organises rows in groups of
  // eight even when the shape reads fewer ("tcgen05.cp" page, "Shared
  // descriptor address walk").  Unswizzled, a group is an 8 x 16-byte block
  // per 16-byte column (columns LDO apart); swizzled, 8 rows of 16 << mode
  // bytes, whose swizzle stays inside the period-aligned blocks it spans.
  // Decompression keeps the base shape's source footprint.
  const int base_shape = shape % 4;
  const uint32_t rows = base_shape == 2 ? 32u : base_shape == 3 ? 4u : 128u;
  const uint32_t words = base_shape == 0 || base_shape == 3 ? 8u : 4u;
  const uint32_t groups = (rows + 7) / 8;
  const uint32_t columns = swizzle == 0 ? (words + 3) / 4 : 1u;
  const uint32_t block = 8u * (16u << swizzle);
  const uint32_t span = origin_bytes + (groups - 1) * sdo + (columns - 1) * (swizzle == 0 ? ldo : 0u) + block;
  const uint32_t period = swizzle_period(swizzle);
  if ((span + period - 1) / period * period > static_cast<uint32_t>(image_words) * 4u) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + static_cast<size_t>(image_words) * 4;
  cudaError_t e = cudaFuncSetAttribute(probe_cp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  probe_cp_kernel<<<1, 128, smem, as_stream(stream)>>>(image, image_words, shape, origin_bytes,
                                                       sdesc_hi(ldo, sdo, swizzle), out, device_error_word(dev),
                                                       wait_timeout_ns());
  return finish_launch(1);
}

extern "C" int tcg_probe_ld_shape(const uint32_t* in, int shape, int num, int half, uint32_t* out, void* stream) {
  if (!in || !out || shape < 0 || shape > 3 || (half != 0 && half != 1)) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaStream_t s = as_stream(stream);
#define TCG_LD_CASE(SH, NU) \
  if (shape == SH && num == NU) { probe_ld_shape_kernel<SH, NU><<<1, 128, 0, s>>>(in, half, out); return finish_launch(1); }
  // every repeat count whose columns fit the 32-column image
  TCG_LD_CASE(0, 1) TCG_LD_CASE(0, 2) TCG_LD_CASE(0, 4) TCG_LD_CASE(0, 8) TCG_LD_CASE(0, 16) TCG_LD_CASE(0, 32)
  TCG_LD_CASE(1, 1) TCG_LD_CASE(1, 2) TCG_LD_CASE(1, 4) TCG_LD_CASE(1, 8) TCG_LD_CASE(1, 16)
  TCG_LD_CASE(2, 1) TCG_LD_CASE(2, 2) TCG_LD_CASE(2, 4) TCG_LD_CASE(2, 8)
  TCG_LD_CASE(3, 1) TCG_LD_CASE(3, 2) TCG_LD_CASE(3, 4)
#undef TCG_LD_CASE
  return TCG_ERR_INVALID;
}

extern "C" int tcg_probe_mma_tile(const void* A, const void* B, int N, int K, int is_bf16, float* D, void* stream) {
  if (!A || !B || !D || N < 16 || N > 256 || N % 16 || K < 16 || K > 64 || K % 16) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + (128 + 256) * 128;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  const uint32_t idesc = idesc_f16(is_bf16 != 0, true, false, false, 128, N);
  probe_mma_tile_kernel<<<1, 128, smem, as_stream(stream)>>>(static_cast<const uint16_t*>(A),
                                                             static_cast<const uint16_t*>(B), N, K, idesc, 0, D,
                                                             device_error_word(dev), wait_timeout_ns());
  return finish_launch(1);
}

extern "C" int tcg_probe_mma_tmem_a(const void* A, const void* B, int N, int K, int is_bf16, float* D, void* stream) {
  if (!A || !B || !D || N < 16 || N > 256 || N % 16 || K < 16 || K > 64 || K % 16) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + 256 * 128;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_tmem_a_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  const uint32_t idesc = idesc_f16(is_bf16 != 0, true, false, false, 128, N);
  probe_mma_tmem_a_kernel<<<1, 128, smem, as_stream(stream)>>>(static_cast<const uint16_t*>(A),
                                                               static_cast<const uint16_t*>(B), N, K, idesc, D,
                                                               device_error_word(dev), wait_timeout_ns());
  return finish_launch(1);
}

extern "C" int tcg_probe_mma_ws64(const void* A, int a_tmem, const void* B, int N, int K, int is_bf16, uint32_t* out,
                                  void* stream) {
  if (!A || !B || !out || (N != 64 && N != 128 && N != 256) || K < 16 || K > 64 || K % 16) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + (128 + 256) * 128;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_ws64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  const uint32_t idesc = idesc_f16(is_bf16 != 0, true, false, false, 64, N);
  probe_mma_ws64_kernel<<<1, 128, smem, as_stream(stream)>>>(static_cast<const uint16_t*>(A),
                                                             static_cast<const uint16_t*>(B), N, K, a_tmem ? 1 : 0,
                                                             idesc, out, device_error_word(dev), wait_timeout_ns());
  return finish_launch(1);
}

extern "C" int tcg_probe_mma_tile_ws(const void* A, const void* B, int N, int K, int is_bf16, float* D,
                                     void* stream) {
  if (!A || !B || !D || (N != 64 && N != 128 && N != 256) || K < 16 || K > 64 || K % 16) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + (128 + 256) * 128;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  const uint32_t idesc = idesc_f16(is_bf16 != 0, true, false, false, 128, N);
  probe_mma_tile_kernel<<<1, 128, smem, as_stream(stream)>>>(static_cast<const uint16_t*>(A),
                                                             static_cast<const uint16_t*>(B), N, K, idesc, 1, D,
                                                             device_error_word(dev), wait_timeout_ns());
  return finish_launch(1);
}

namespace {

// Largest distance past an issue's descriptor origin that its walk can reach
// for an operand of `rows_mn` M/N rows: under the pages' assignment of LDO and
// SDO and under the swapped one (so that a misreading still stays inside the
// operand's region), plus the whole row-group block it lands in.
uint32_t image_walk_reach(tcg_major major, int swizzle, int rows_mn, int esize, uint32_t ldo, uint32_t sdo) {
  const uint32_t krows = 32u / static_cast<uint32_t>(esize);  // K per issue: 16 (16-bit), 8 (TF32)
  uint32_t groups, chunks, block;
  if (major == TCG_K_MAJOR) {
    groups = (static_cast<uint32_t>(rows_mn) + 7u) / 8u;
    chunks = swizzle == 0 ? 2u : 1u;  // 32 bytes of K: two 16-byte chunks unswizzled
    block = swizzle == 0 ? 128u : 8u * (16u << swizzle);
  } else {
    const uint32_t rb = swizzle == 4 ? 128u : (16u << swizzle);
    const uint32_t g = swizzle == 4 ? 4u : 8u;
    groups = (krows + g - 1u) / g;
    chunks = (static_cast<uint32_t>(rows_mn * esize) + rb - 1u) / rb;
    block = g * rb;
  }
  const uint32_t r1 = (groups - 1u) * ldo + (chunks - 1u) * sdo;
  const uint32_t r2 = (groups - 1u) * sdo + (chunks - 1u) * ldo;
  return (r1 > r2 ? r1 : r2) + block;
}

int image_operand(const tcg_probe_operand* o, int rows_mn, int esize, bool tf32, int ksteps, ImageOperand* out) {
  if (!o || !o->image || reinterpret_cast<uintptr_t>(o->image) % 16) return TCG_ERR_INVALID;
  if (o->bytes <= 0 || o->bytes % 16 || static_cast<uint32_t>(o->bytes) > MMA_IMAGE_REGION) return TCG_ERR_INVALID;
  if (o->major != TCG_K_MAJOR && o->major != TCG_MN_MAJOR) return TCG_ERR_INVALID;
  if (o->swizzle < 0 || o->swizzle > 4) return TCG_ERR_INVALID;
  // "swizzle=4" is the 32-bit MN-major mode; TF32 MN-major takes no other
  if ((o->swizzle == 4) != (tf32 && o->major == TCG_MN_MAJOR)) return TCG_ERR_UNSUPPORTED;
  if ((o->ldo | o->sdo) & 15u || o->ldo >= (1u << 18) || o->sdo >= (1u << 18)) return TCG_ERR_INVALID;
  const uint32_t reach = image_walk_reach(o->major, o->swizzle, rows_mn, esize, o->ldo, o->sdo);
  for (int j = 0; j < ksteps; ++j) {
    if (o->start[j] & 15u) return TCG_ERR_INVALID;
    // the walk, a swizzle period of slack and the whole block stay in the region
    if (static_cast<uint64_t>(o->start[j]) + reach + 1024u > MMA_IMAGE_REGION) return TCG_ERR_INVALID;
  }
  out->image = static_cast<const uint4*>(o->image);
  out->words16 = o->bytes / 16;
  out->desc_hi = sdesc_hi(o->ldo, o->sdo, o->swizzle);
  for (int j = 0; j < 8; ++j) out->start[j] = j < ksteps ? o->start[j] : 0u;
  return TCG_OK;
}

}  // namespace

extern "C" int tcg_probe_mma_image(const tcg_probe_operand* a, const tcg_probe_operand* b, tcg_input in_type, int N,
                                   int ksteps, float* D, void* stream) {
  if (!D || N < 16 || N > 256 || N % 16 || ksteps < 1 || ksteps > 8) return TCG_ERR_INVALID;
  if (in_type != TCG_IN_F16 && in_type != TCG_IN_BF16 && in_type != TCG_IN_TF32) return TCG_ERR_INVALID;
  const bool tf32 = in_type == TCG_IN_TF32;
  const int esize = tf32 ? 4 : 2;
  ImageOperand ia, ib;
  if (int rc = image_operand(a, 128, esize, tf32, ksteps, &ia)) return rc;
  if (int rc = image_operand(b, N, esize, tf32, ksteps, &ib)) return rc;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const size_t smem = 1024 + 2 * static_cast<size_t>(MMA_IMAGE_REGION);
  cudaError_t e = cudaFuncSetAttribute(probe_mma_image_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return record_cuda(e);
  const bool a_mn = a->major == TCG_MN_MAJOR, b_mn = b->major == TCG_MN_MAJOR;
  const uint32_t idesc = tf32 ? idesc_tf32(a_mn, b_mn, 128, N) : idesc_f16(in_type == TCG_IN_BF16, true, a_mn, b_mn, 128, N);
  probe_mma_image_kernel<<<1, 128, smem, as_stream(stream)>>>(ia, ib, tf32 ? 1 : 0, idesc, N, ksteps, D,
                                                              device_error_word(dev), wait_timeout_ns());
  return finish_launch(1);
}

extern "C" int tcg_probe_ld_split(const uint32_t* in, int num, int imm_lanes, int imm_cols, uint32_t* out_ld,
                                  uint32_t* out_st, void* stream) {
  if (!in || !out_ld || !out_st) return TCG_ERR_INVALID;
  const bool num_ok = num == 1 || num == 2 || num == 4 || num == 8;
  const bool imm_ok = (imm_lanes == 16 && (imm_cols == 0 || imm_cols == 8 || imm_cols == 16)) ||
                      (imm_lanes == 0 && imm_cols == 16);
  if (!num_ok || !imm_ok) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaStream_t s = as_stream(stream);
#define TCG_SPLIT_CASE(NU, IL, IC)                                                                        \
  if (num == NU && imm_lanes == IL && imm_cols == IC) {                                                  \
    probe_split_kernel<NU, (static_cast<uint32_t>(IL) << 16) + IC><<<1, 128, 0, s>>>(in, out_ld, out_st); \
    return finish_launch(1);                                                                             \
  }
#define TCG_SPLIT_NUMS(IL, IC) \
  TCG_SPLIT_CASE(1, IL, IC) TCG_SPLIT_CASE(2, IL, IC) TCG_SPLIT_CASE(4, IL, IC) TCG_SPLIT_CASE(8, IL, IC)
  TCG_SPLIT_NUMS(16, 8) TCG_SPLIT_NUMS(16, 0) TCG_SPLIT_NUMS(0, 16) TCG_SPLIT_NUMS(16, 16)
#undef TCG_SPLIT_NUMS
#undef TCG_SPLIT_CASE
  return TCG_ERR_INVALID;
}

extern "C" int tcg_probe_stmatrix(const uint32_t* regs, const uint32_t* row_off, int count, int trans, uint32_t* out,
                                  void* stream) {
  if (!regs || !row_off || !out) return TCG_ERR_INVALID;
  if (count != 1 && count != 2 && count != 4) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaStream_t s = as_stream(stream);
  if (count == 1 && !trans) probe_stmatrix_kernel<1, false><<<1, 32, 0, s>>>(regs, row_off, out);
  else if (count == 1) probe_stmatrix_kernel<1, true><<<1, 32, 0, s>>>(regs, row_off, out);
  else if (count == 2 && !trans) probe_stmatrix_kernel<2, false><<<1, 32, 0, s>>>(regs, row_off, out);
  else if (count == 2) probe_stmatrix_kernel<2, true><<<1, 32, 0, s>>>(regs, row_off, out);
  else if (count == 4 && !trans) probe_stmatrix_kernel<4, false><<<1, 32, 0, s>>>(regs, row_off, out);
  else if (count == 4) probe_stmatrix_kernel<4, true><<<1, 32, 0, s>>>(regs, row_off, out);
  else return TCG_ERR_INVALID;
  return finish_launch(1);
}

extern "C" int tcg_probe_ldmatrix_x2(const uint32_t* x, uint32_t* out, void* stream) {
  if (!x || !out) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  probe_ldmatrix_kernel<<<1, 32, 0, as_stream(stream)>>>(x, out);
  return finish_launch(1);
}

extern "C" int tcg_probe_wait_timeout(uint64_t timeout_ns, void* stream) {
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  if (timeout_ns < 1000) timeout_ns = 1000;
  if (timeout_ns > 10000000000ull) timeout_ns = 10000000000ull;
  probe_wait_timeout_kernel<<<1, 32, 0, as_stream(stream)>>>(device_error_word(dev), timeout_ns);
  return finish_launch(1);
}
