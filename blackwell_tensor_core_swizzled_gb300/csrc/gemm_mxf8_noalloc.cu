// Block-scaled MXFP8 GEMM that allocates no device memory.
//
// tcg_gemm_mxf8_blockscaled needs a scratch buffer for the rearranged scale
// factors and grows one per (device, stream) with cudaMalloc / cudaFree.
// Some callers cannot allow that: a framework whose caching allocator owns
// every byte of device memory and forbids anyone else to call cudaMalloc, or
// code that must not stall, since replacing a too-small buffer calls
// cudaFree, which waits for the whole device.  For them this entry point keeps
// its scratch in one fixed array that is part of the library's device image
// (every GPU that loads the library holds it until the process exits).
//
// Limits and sharing:
//  * the two scale images of one call must fit in kScratchBytes (16 MiB;
//    an 8192 x 8192 x 8192 problem needs 4 MiB); larger problems are
//    rejected with TCG_ERR_UNSUPPORTED.  Every argument (sizes, pointers,
//    alignment, output and accumulator types, the device) is checked before
//    anything is queued, so a call that fails leaves the array untouched;
//  * every call on every stream of a device uses the same array, which keeps
//    the previous call's contents.  Each call rewrites every byte of the image
//    region it reads (padding included), so nothing needs clearing, but calls
//    whose work overlaps on the GPU (different streams without ordering
//    between them) race on the array: order them.
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.h"
#include "tcg.h"

namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(16) << 20;

static __device__ __align__(256) uint8_t g_mxf8_scale_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array for the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in,
// never a device address.
int scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return TCG_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lk(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_mxf8_scale_scratch);
    if (e != cudaSuccess) return tcg::record_cuda(e);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TCG_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int tcg_gemm_mxf8_blockscaled_noalloc(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major,
                                                 int64_t lda, const void* B, tcg_major b_major, int64_t ldb,
                                                 const uint8_t* SFA, const uint8_t* SFB, void* D, tcg_dtype d_type,
                                                 int64_t ldd, tcg_dtype acc_type, void* stream) {
  if (M < 0 || N < 0 || K < 0) return TCG_ERR_INVALID;
  if (M == 0 || N == 0) return TCG_OK;
  if (acc_type != TCG_F32) return TCG_ERR_UNSUPPORTED;
  if (K == 0)  // D = 0; no scale images are needed
    return tcg_gemm_mxf8_blockscaled(M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type,
                                     stream);
  if (!A || !B || !D || !SFA || !SFB) return TCG_ERR_INVALID;
  if (d_type != TCG_F32 && d_type != TCG_F16 && d_type != TCG_BF16) return TCG_ERR_INVALID;
  if (ldd == 0) ldd = N;
  if (ldd < N) return TCG_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(D) % (d_type == TCG_F32 ? 4 : 2)) return TCG_ERR_ALIGNMENT;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return TCG_ERR_UNSUPPORTED;
  if (a_major != TCG_K_MAJOR && a_major != TCG_MN_MAJOR) return TCG_ERR_INVALID;
  if (b_major != TCG_K_MAJOR && b_major != TCG_MN_MAJOR) return TCG_ERR_INVALID;
  // operand checks before anything is queued (E4M3: one byte per element)
  const int64_t a_inner = a_major == TCG_K_MAJOR ? K : M;
  const int64_t b_inner = b_major == TCG_K_MAJOR ? K : N;
  if (lda == 0) lda = a_inner;
  if (ldb == 0) ldb = b_inner;
  if (lda < a_inner || ldb < b_inner) return TCG_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) % 16 || lda % 16 || ldb % 16)
    return TCG_ERR_ALIGNMENT;

  const int tile_n = tcg_mxf8_tile_n(M, N, K, b_major, 0);
  if (tile_n < 0) return tile_n;
  const int64_t bytes_a = tcg_mxf8_scale_image_bytes(M, K, 128);
  const int64_t bytes_b = tcg_mxf8_scale_image_bytes(N, K, tile_n);
  if (bytes_a < 0 || bytes_b < 0) return TCG_ERR_INVALID;
  if (static_cast<uint64_t>(bytes_a + bytes_b) > kScratchBytes) {
    tcg::set_error_message("scale images exceed the 16 MiB no-allocation scratch array");
    return TCG_ERR_UNSUPPORTED;
  }

  int dev = 0;
  if (int rc = tcg::current_device_checked(&dev)) return rc;  // an sm_103 device is current
  void* scratch = nullptr;
  if (int rc = scratch_address(dev, &scratch)) return rc;
  uint8_t* img_a = static_cast<uint8_t*>(scratch);
  uint8_t* img_b = img_a + cdiv(bytes_a, 256) * 256;  // both images 256-byte aligned

  // both images in one launch, then the GEMM reads them
  if (int rc = tcg_mxf8_prepare_scales_ab(SFA, M, img_a, SFB, N, tile_n, img_b, K, stream)) return rc;
  tcg_gemm_args args;
  std::memset(&args, 0, sizeof args);
  args.M = M;
  args.N = N;
  args.K = K;
  args.in_type = TCG_IN_E4M3;
  args.A = A;
  args.a_major = a_major;
  args.lda = lda;
  args.B = B;
  args.b_major = b_major;
  args.ldb = ldb;
  args.SFA_img = img_a;
  args.SFB_img = img_b;
  args.D = D;
  args.d_type = d_type;
  args.ldd = ldd;
  args.acc_type = acc_type;
  args.split_k = 1;  // split-K would need the library's (allocated) workspace
  if (int rc = tcg_gemm(&args, stream)) return rc;
  tcg::set_launch_count(2);
  return TCG_OK;
}
