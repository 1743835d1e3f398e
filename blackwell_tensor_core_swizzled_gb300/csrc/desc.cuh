// Shared-memory descriptors and instruction descriptors for tcgen05.
//
// The byte walk a descriptor encodes is the one the Apache TVM TIRx
// "tcgen05.cp" page gives ("Shared descriptor address walk"): row r starts
// at (r//8)*SDO + (r%8)*(16 << swizzle) bytes from the origin, an unswizzled
// word w adds (w//4)*LDO + (w%4)*4, swizzled words are contiguous.  The
// "tcgen05.mma" page ("Shared descriptors are byte-stride contracts") fixes
// which stride is which per operand majorness, and its "swizzle=4" section
// the 128-byte-span / 32-byte-atom mode used by MN-major 32-bit operands.
//
// The pages give the walk, not the bit encoding.  The 64-bit layout below is
// the PTX ISA's tcgen05 shared memory descriptor: start address >> 4 in bits
// [0,14), leading-dimension byte offset >> 4 in [16,30), stride-dimension
// byte offset >> 4 in [32,46), the fixed version value 1 at bit 46, base
// offset [49,52) (0: every base here is period aligned), and the swizzle
// layout type in [61,64).  The start address is the un-swizzled (logical)
// address of the origin ("tcgen05.mma" page: the origin is inverse-swizzled
// before encoding so that it is not permuted twice).
#pragma once

#include <cstdint>

namespace tcg {

// The pages' logical swizzle modes.
enum SwizzleMode : int { SW_NONE = 0, SW_32B = 1, SW_64B = 2, SW_128B = 3, SW_128B_ATOM32 = 4 };

// Descriptor layout-type field for each logical mode.
__host__ __device__ constexpr uint32_t layout_type_field(int mode) {
  return mode == SW_NONE ? 0u : mode == SW_32B ? 6u : mode == SW_64B ? 4u : mode == SW_128B ? 2u : 1u;
}

__host__ __device__ constexpr uint32_t swizzle_period(int mode) {
  return mode == SW_NONE ? 16u : mode == SW_32B ? 256u : mode == SW_64B ? 512u : mode == SW_128B ? 1024u : 512u;
}

// Physical shared byte address of a logical one under a swizzle mode (used
// where ordinary stores must build an image that a descriptor reads, e.g.
// the layout probes).  Modes 1..3 XOR the 16-byte chunk index with address
// bits from bit 7 upward; mode 4 is offset ^ ((offset >> 2) & 96).
__host__ __device__ constexpr uint32_t swizzle_addr(uint32_t a, int mode) {
  return mode == SW_NONE ? a
         : mode == SW_128B_ATOM32 ? (a ^ ((a >> 2) & 96u))
                                  : (a ^ ((a >> 3) & ((((1u << mode) - 1u)) << 4)));
}

// Everything of a shared descriptor except the start address.
__host__ __device__ constexpr uint64_t sdesc_hi(uint32_t ldo_bytes, uint32_t sdo_bytes, int mode) {
  return (static_cast<uint64_t>((ldo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sdo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (static_cast<uint64_t>(layout_type_field(mode)) << 61);
}

// Full descriptor for a shared::cta byte address.
__host__ __device__ constexpr uint64_t sdesc(uint32_t smem_addr, uint64_t hi) {
  return hi | static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
}

// Host-side validation of a descriptor's fields ("tcgen05.cp" page: strides
// are non-negative 16-byte multiples below 2^18, origins 16-byte aligned,
// swizzled bases aligned to the mode's period).  Returns true if valid.
inline bool sdesc_fields_ok(uint32_t origin, uint32_t ldo, uint32_t sdo, int mode, uint32_t base) {
  if (mode < 0 || mode > 4) return false;
  if ((ldo & 15u) || (sdo & 15u) || ldo >= (1u << 18) || sdo >= (1u << 18)) return false;
  if (origin & 15u) return false;
  if (mode != SW_NONE && (base % swizzle_period(mode)) != 0) return false;
  return true;
}

// ---------------------------------------------------------------------------
// Instruction descriptors (32-bit), PTX ISA tcgen05 "Instruction descriptor"
// tables.  kind::f16 / kind::tf32: D format [4,6) (0 F16, 1 F32), A format
// [7,10), B format [10,13) (kind::f16: 0 F16, 1 BF16; kind::tf32: 2 TF32),
// transpose (MN-major) A bit 15, B bit 16, N>>3 in [17,23), M>>4 in [24,29).
// kind::mxf8f6f4 block-scaled: SFB id [4,6), A/B formats (E4M3 0, E5M2 1,
// E2M3 3, E3M2 4, E2M1 5), majors, N>>3, scale type bit 23 (1 = UE8M0), M>>4,
// SFA id [29,31).
// ---------------------------------------------------------------------------

__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool d_f32, bool a_mn, bool b_mn, int M, int N) {
  return (static_cast<uint32_t>(d_f32) << 4) | (static_cast<uint32_t>(bf16) << 7) |
         (static_cast<uint32_t>(bf16) << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__host__ __device__ constexpr uint32_t idesc_tf32(bool a_mn, bool b_mn, int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// kind::mxf8f6f4 operand format codes (A bits [7,10), B bits [10,13)).
enum MxFormat : uint32_t { MXF_E4M3 = 0, MXF_E5M2 = 1, MXF_E2M3 = 3, MXF_E3M2 = 4, MXF_E2M1 = 5 };

__host__ __device__ constexpr uint32_t idesc_mxf8(bool a_mn, bool b_mn, int M, int N, uint32_t a_fmt = MXF_E4M3,
                                                  uint32_t b_fmt = MXF_E4M3) {
  return (a_fmt << 7) | (b_fmt << 10) | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

// kind::mxf4 / kind::mxf4nvf4: A and B are E2M1 (code 1), K-major; bit 23 the
// scale type (1 UE8M0 for scale_vec::2X, 0 UE4M3 for scale_vec::4X); bit 31
// (K = 96 for sparse forms) stays 0 for K = 64.
__host__ __device__ constexpr uint32_t idesc_fp4(int M, int N, bool ue8m0) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(ue8m0) << 23) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Scale-factor ids: which byte of the 32-bit scale column each operand's
// scales are read from.
__host__ __device__ constexpr uint32_t idesc_sf_ids(uint32_t sfa_id, uint32_t sfb_id) {
  return ((sfb_id & 3u) << 4) | ((sfa_id & 3u) << 29);
}

}  // namespace tcg
