// Host side of the C ABI declared in include/tcg.h: argument validation, TMA
// tensor-map encoding, tile/variant selection, launches, the per-device error
// word and the block-scale workspace.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include "common.h"
#include "gemm_chain.cuh"
#include "gemm_kernel.cuh"

namespace tcg {

// Per-device error word: a kernel whose bounded wait runs out writes a code
// here (see ErrSite); tcg_check() reads and clears it.
__device__ unsigned long long g_error_word;

namespace {

thread_local std::string t_last_error;
thread_local int t_last_launches = 0;
// The last call's plan, formatted only when tcg_last_plan_string asks for it
// (formatting on every call measured a quarter of a microsecond).
struct PlanRecord {
  bool valid = false;
  bool k_zero = false;
  int cg = 0, bn = 0, clusters = 0, split = 0;
  int mc = 1;  // CTAs per cluster sharing B tiles by multicast
  bool swapped = false, stream_k = false, frag = false;
};
thread_local PlanRecord t_plan;
thread_local std::string t_last_plan;
// phase trace requested for the next GEMM launch on this thread
thread_local unsigned long long* t_trace_buf = nullptr;
thread_local int t_trace_ctas = 0;
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool init = false;
  bool usable = false;
  int sms = 0;
  unsigned long long* err = nullptr;
  // per kernel host stub: smem attribute set, max co-resident clusters
  std::map<const void*, int> max_clusters;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_get = nullptr;
std::once_flag g_ctx_get_once;

struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Split-K / stream-K workspace per (device, stream): fp32 partial-tile slots,
// written by the GEMM and read by the reduction kernel that follows it on the
// same stream (their contents never need clearing).
struct SplitWorkspace {
  void* slots = nullptr;
  size_t slot_bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, SplitWorkspace> g_split_ws;

void load_timeout_env() {
  static std::once_flag once;
  std::call_once(once, [] {
    if (const char* v = std::getenv("TCG_WAIT_TIMEOUT_NS")) {
      const unsigned long long ns = std::strtoull(v, nullptr, 10);
      if (ns > 0) g_timeout_ns.store(ns < 1000 ? 1000 : ns);
    }
  });
}

DeviceState* device_state(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
      cudaGetLastError();
      return &d;
    }
    d.sms = prop.multiProcessorCount;
    d.usable = (prop.major == 10 && prop.minor == 3);
    void* p = nullptr;
    if (d.usable && cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) {
      d.err = static_cast<unsigned long long*>(p);
      cudaMemset(d.err, 0, sizeof(unsigned long long));
    } else {
      cudaGetLastError();
      d.usable = false;
    }
  }
  return &d;
}

int encode_ready() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  return g_encode ? TCG_OK : TCG_ERR_CUDA;
}

// Encoded tensor maps, per host thread: a map is a pure function of its
// encode arguments (data type, base address, extents, strides, box, swizzle),
// so a map found under the same arguments is the map the driver would return
// again.  A 64-slot direct-mapped table keyed by an FNV-1a hash of the
// arguments; a colliding key replaces the slot.  Per thread, so no lock.
struct MapKey {
  uint64_t base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  uint32_t dt, rank, sw;
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int kMapSlots = 64;
thread_local MapSlot t_maps[kMapSlots];

uint64_t map_key_hash(const MapKey& k) {
  const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof k; ++i) h = (h ^ p[i]) * 1099511628211ull;
  return h;
}

int encode_map(CUtensorMap* map, const MapKey& key, CUtensorMapDataType dt, void* base, const cuuint64_t* dims,
               const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  MapSlot& slot = t_maps[map_key_hash(key) % kMapSlots];
  if (slot.used && std::memcmp(&slot.key, &key, sizeof key) == 0) {
    *map = slot.map;
    return TCG_OK;
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, dt, key.rank, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return static_cast<int>(r);
  slot.key = key;
  slot.map = *map;
  slot.used = true;
  return TCG_OK;
}

// 2-D tiled tensor map over a row-major matrix: `inner` elements per row
// (contiguous), `outer` rows, `ld` elements between rows.
int make_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  if (encode_ready() != TCG_OK) {
    t_last_error = "cuTensorMapEncodeTiled entry point unavailable";
    return TCG_ERR_CUDA;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {ld * static_cast<uint64_t>(esize)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.base = reinterpret_cast<uint64_t>(base);
  key.dims[0] = inner;
  key.dims[1] = outer;
  key.strides[0] = strides[0];
  key.box[0] = box_inner;
  key.box[1] = box_outer;
  key.dt = static_cast<uint32_t>(dt);
  key.rank = 2;
  key.sw = static_cast<uint32_t>(sw);
  const int r = encode_map(map, key, dt, const_cast<void*>(base), dims, strides, box, sw);
  if (r != TCG_OK) {
    char buf[160];
    std::snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d): dims %llu x %llu, ld %llu, box %u x %u",
                  static_cast<int>(r), static_cast<unsigned long long>(inner),
                  static_cast<unsigned long long>(outer), static_cast<unsigned long long>(ld), box_inner, box_outer);
    t_last_error = buf;
    return TCG_ERR_CUDA;
  }
  return TCG_OK;
}

// 3D map over a dense [outer][mid][inner] array (row strides inner*esize and
// mid*inner*esize bytes).
int make_map_3d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int esize, uint64_t inner,
                uint64_t mid, uint64_t outer, uint32_t box_inner, uint32_t box_mid, CUtensorMapSwizzle sw) {
  if (encode_ready() != TCG_OK) {
    t_last_error = "cuTensorMapEncodeTiled entry point unavailable";
    return TCG_ERR_CUDA;
  }
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * static_cast<uint64_t>(esize), inner * mid * static_cast<uint64_t>(esize)};
  const cuuint32_t box[3] = {box_inner, box_mid, 1};
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.base = reinterpret_cast<uint64_t>(base);
  for (int i = 0; i < 3; ++i) key.dims[i] = dims[i];
  key.strides[0] = strides[0];
  key.strides[1] = strides[1];
  key.box[0] = box_inner;
  key.box[1] = box_mid;
  key.box[2] = 1;
  key.dt = static_cast<uint32_t>(dt);
  key.rank = 3;
  key.sw = static_cast<uint32_t>(sw);
  const int r = encode_map(map, key, dt, const_cast<void*>(base), dims, strides, box, sw);
  if (r != TCG_OK) {
    t_last_error = "cuTensorMapEncodeTiled (3D) failed (" + std::to_string(static_cast<int>(r)) + ")";
    return TCG_ERR_CUDA;
  }
  return TCG_OK;
}

// Block-scaled formats.  E4M3 / E5M2 bytes and the FP6 formats (packed in
// global memory) run on kind::mxf8f6f4 with one byte of shared memory per
// element (TMA expands FP6 into 16-byte blocks of sixteen values and padding,
// the layout the "tcgen05.cp" page's FP4 / FP6 shapes describe).  FP4 (E2M1
// with e8m0 scales per 32, or the NVFP4 form with unsigned E4M3 scales per 16)
// stays packed, two values per byte, on kind::mxf4 / kind::mxf4nvf4.
bool is_mx(tcg_input t) {
  return t == TCG_IN_E4M3 || t == TCG_IN_E5M2 || t == TCG_IN_E3M2 || t == TCG_IN_E2M3 || t == TCG_IN_E2M1 ||
         t == TCG_IN_NVF4;
}
bool is_fp6(tcg_input t) { return t == TCG_IN_E3M2 || t == TCG_IN_E2M3; }
bool is_fp4(tcg_input t) { return t == TCG_IN_E2M1 || t == TCG_IN_NVF4; }
int bits_of(tcg_input t) {
  return t == TCG_IN_TF32 ? 32 : is_fp4(t) ? 4 : is_fp6(t) ? 6 : is_mx(t) ? 8 : 16;
}
// bytes per element in shared memory (and in global memory for unpacked
// types); packed FP4 is half a byte and handled by its own branches
int esize_of(tcg_input t) { return t == TCG_IN_TF32 ? 4 : is_mx(t) ? 1 : 2; }
// K elements per ring stage: one 128-byte shared row (packed FP4: 256)
int stage_k(tcg_input t) { return is_fp4(t) ? 256 : 128 / esize_of(t); }
// global bytes of `ld` elements
int64_t row_bytes(tcg_input t, int64_t ld) { return ld * bits_of(t) / 8; }
// bytes TMA writes per operand row per stage: the packed FP6 types write only
// their data bytes (96 per 128 elements) and skip the padding of each block
int stage_row_tx(tcg_input t) { return is_fp6(t) ? 96 : 128; }
uint32_t mx_format(tcg_input t) {
  return t == TCG_IN_E5M2 ? MXF_E5M2 : t == TCG_IN_E3M2 ? MXF_E3M2 : t == TCG_IN_E2M3 ? MXF_E2M3 : MXF_E4M3;
}
int dsize_of(tcg_dtype t) { return t == TCG_F32 ? 4 : 2; }

// Validates one operand; fills its leading dimension when 0 (packed).
// Packed 6- and 4-bit operands are K-major, K a multiple of 128, with 32-byte
// aligned bases and row strides (the TMA rules of the padded element types).
int check_operand(const void* ptr, tcg_major major, int64_t mn, int64_t K, int64_t* ld, tcg_input t) {
  if (major != TCG_K_MAJOR && major != TCG_MN_MAJOR) return TCG_ERR_INVALID;
  const int64_t inner = major == TCG_K_MAJOR ? K : mn;
  if (*ld == 0) *ld = inner;
  if (*ld < inner || *ld < 1) return TCG_ERR_INVALID;
  if (!ptr) return TCG_ERR_INVALID;
  if (is_fp6(t)) {
    if (major != TCG_K_MAJOR) return TCG_ERR_UNSUPPORTED;
    if (K % 128 || (*ld * bits_of(t)) % 8) return TCG_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(ptr) % 32 || row_bytes(t, *ld) % 32) return TCG_ERR_ALIGNMENT;
    return TCG_OK;
  }
  if (is_fp4(t)) {  // packed bytes: 16-byte aligned rows of K/2 bytes
    if (major != TCG_K_MAJOR) return TCG_ERR_UNSUPPORTED;
    if (K % 32 || *ld % 32) return TCG_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(ptr) % 16) return TCG_ERR_ALIGNMENT;
    return TCG_OK;
  }
  if (reinterpret_cast<uintptr_t>(ptr) % 16) return TCG_ERR_ALIGNMENT;
  if ((*ld * esize_of(t)) % 16) return TCG_ERR_ALIGNMENT;
  return TCG_OK;
}

struct Plan {
  KernelInfo ki;
  int cta_group;
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int pick_cta_group(const tcg_gemm_args& a) {
  if (a.cta_group == 1 || a.cta_group == 2) return a.cta_group;
  // pairs halve the B traffic per SM and each MMA issue covers 256 rows; they
  // win from the first problem taller than one 128-row tile (bf16 x 8192 x
  // 8192, single CTAs vs pairs: 160 rows 64.2 / 56.0 us, 256 rows 64.2 / 53.9,
  // 768 rows 105.1 / 88.7; 512 x 4096 x 4096 35.5 / 29.4)
  return (a.M > 128 && a.N >= 1024) ? 2 : 1;
}

// Packed-FP4 CTA pairs on many tiles: 256 x 384 tiles (two MMAs per K step,
// N = 256 and N = 128).  Each SM then takes in 320 rows of operands per
// 128 x 384 outputs instead of 256 per 128 x 256, a sixth fewer bytes per
// product, and 8 (MXFP4) or 16 (NVFP4) scale copies per 384 columns instead
// of 6 or 12 per 256.  Measured at 8192^3: MXFP4 +3.5 %, NVFP4 +1 %; for
// MXFP8 and FP6 the same tile lost 0.7 % (and 1 % as two N = 192 MMAs), so
// those keep 256 x 256.
// The rule depends on the format and shape alone, so that scale images
// prepared for tcg_tile_n always match.
bool wide_tiles(const tcg_gemm_args& a, int cg) {
  return is_fp4(a.in_type) && cg == 2 && a.b_major == TCG_K_MAJOR && cdiv(a.M, 256) * cdiv(a.N, 384) >= 300;
}

int get_plan(const tcg_gemm_args& a, Plan* plan) {
  const int cg = pick_cta_group(a);
  plan->cta_group = cg;
  switch (a.in_type) {
    case TCG_IN_F16:
    case TCG_IN_BF16:
      // narrow (N <= 32, K-major B): 32-column tiles; skinny (M <= 128,
      // K-major A): 64-column tiles staging 32, 64 or 128 rows of A
      plan->ki = kinfo_f16(cg, cg != 1                                       ? F16_WIDE
                               : a.N <= 32 && a.b_major == TCG_K_MAJOR       ? F16_NARROW_N
                               : a.M <= 32 && a.a_major == TCG_K_MAJOR       ? F16_SKINNY_M
                               : a.M <= 64 && a.a_major == TCG_K_MAJOR       ? F16_SKINNY_M64
                               : a.M <= 128 && a.a_major == TCG_K_MAJOR      ? F16_SKINNY_M128
                                                                             : F16_WIDE);
      break;
    case TCG_IN_TF32: plan->ki = kinfo_tf32(cg); break;
    case TCG_IN_E4M3:
    case TCG_IN_E5M2:
    case TCG_IN_E3M2:
    case TCG_IN_E2M3: plan->ki = kinfo_mxf8(cg); break;
    case TCG_IN_E2M1: plan->ki = kinfo_fp4(cg, false, wide_tiles(a, cg)); break;
    case TCG_IN_NVF4: plan->ki = kinfo_fp4(cg, true, wide_tiles(a, cg)); break;
    default: return TCG_ERR_INVALID;
  }
  // an MN-major B half tile must be whole 128-byte swizzle spans
  if (a.b_major == TCG_MN_MAJOR && (plan->ki.bn / cg) % (128 / esize_of(a.in_type)) != 0) return TCG_ERR_UNSUPPORTED;
  return TCG_OK;
}

// The variant for a problem on a device with `sms` SMs: get_plan's choice
// refined by the tile counts, and whether to run the transposed product with
// the operands swapped.
int choose_plan(const tcg_gemm_args& a, int sms, Plan* plan, bool* swap_operands) {
  if (int rc = get_plan(a, plan)) return rc;
  const bool f16_kind = a.in_type == TCG_IN_F16 || a.in_type == TCG_IN_BF16;
  const void* f = plan->ki.func;
  // Few rows of A against very many columns of B (decode-like shapes whose
  // 64-column skinny tiles would take more than one wave): compute the
  // transposed product D^T = B^T A^T with the operands' roles swapped, so
  // that B fills the 128-row MMA side (half as many tiles, one pass each); the
  // few rows of A become a 32-column tile and the epilogue stores the result
  // transposed.  Measured on 16-row problems: 16 x 16384 x 4096 35.5 us
  // swapped vs 39.6 us skinny; 16 x 8192 x 8192 38.6 us skinny (128 tiles, one
  // pass) vs 40.6 us swapped (64 tiles: stream-K).  f32 accumulation, single
  // CTAs, K-major A.
  *swap_operands = f16_kind && a.acc_type == TCG_F32 && plan->cta_group == 1 && a.M <= 32 &&
                   a.a_major == TCG_K_MAJOR && cdiv(a.N, 64) > sms;
  // 33..128 rows: the 64-column skinny tiles only while they fit in one wave
  // (128 x 8192 x 8192: 43.6 us vs 47.7 us on 128 x 256 tiles; 128 x 32768 x
  // 4096, 512 skinny tiles: 72.3 us vs 64.1 us)
  if ((f == kinfo_f16(1, F16_SKINNY_M64).func || f == kinfo_f16(1, F16_SKINNY_M128).func) && cdiv(a.N, 64) > sms)
    plan->ki = kinfo_f16(1, F16_WIDE);
  // CTA pairs with few 256 x 256 tiles (at most a quarter of the SMs): 256 x
  // 128 pair tiles, twice as many (back to back, 256 x 4096 x 4096 24.0 ->
  // 19.0 us, 256 x 8192 x 8192 43.1 -> 35 us, 512 x 4096 x 4096 24.2 -> 19.7
  // us; with more tiles the 128-column MMAs' lower efficiency loses: 512 x
  // 8192 x 8192 45.4 -> 60.5 us)
  if (f == kinfo_f16(2, F16_WIDE).func && 4 * cdiv(a.M, 256) * cdiv(a.N, 256) <= sms)
    plan->ki = kinfo_f16(2, F16_PAIR_N128);
  return TCG_OK;
}

int max_clusters_for(DeviceState* d, const KernelInfo& ki, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = d->max_clusters.find(ki.func);
    if (it != d->max_clusters.end()) {
      *out = it->second;
      return TCG_OK;
    }
  }
  cudaError_t e = cudaFuncSetAttribute(ki.func, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem_bytes);
  if (e != cudaSuccess) return record_cuda(e);
  int n = d->sms / ki.cta_group;
  if (ki.cta_group > 1) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(ki.cta_group * n, 1, 1);
    cfg.blockDim = dim3(ki.threads, 1, 1);
    cfg.dynamicSmemBytes = ki.smem_bytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = ki.cta_group;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, ki.func, &cfg);
    if (e == cudaSuccess && clusters > 0)
      n = std::min(n, clusters);
    else
      cudaGetLastError();
  }
  std::lock_guard<std::mutex> lk(g_mu);
  d->max_clusters[ki.func] = n;
  *out = n;
  return TCG_OK;
}

int launch_gemm(const KernelInfo& ki, const GemmParams& prm, int clusters, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ki.cta_group * clusters, 1, 1);
  cfg.blockDim = dim3(ki.threads, 1, 1);
  cfg.dynamicSmemBytes = ki.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (ki.cta_group > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = ki.cta_group;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  // programmatic dependent launch: the kernel's prologue overlaps the tail of
  // the previous kernel on the stream (it waits with griddepcontrol.wait
  // before any global access); back-to-back bf16 8192^3 GEMMs 574.9 ->
  // 567.0 us, 256 x 8192 x 8192 45.2 -> 42.7 us
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  void* args[] = {const_cast<GemmParams*>(&prm)};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, ki.func, args);
  if (e != cudaSuccess) return record_cuda(e);
  return TCG_OK;
}

int workspace(int dev, cudaStream_t s, size_t bytes, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  Workspace& w = g_ws[std::make_pair(dev, s)];
  if (w.bytes < bytes) {
    if (w.ptr) {
      cudaError_t e = cudaFree(w.ptr);  // synchronises: no queued kernel still reads it
      w.ptr = nullptr;
      w.bytes = 0;
      if (e != cudaSuccess) return record_cuda(e);
    }
    const size_t want = std::max(bytes, static_cast<size_t>(1) << 20);
    cudaError_t e = cudaMalloc(&w.ptr, want);
    if (e != cudaSuccess) return record_cuda(e);
    w.bytes = want;
  }
  *out = w.ptr;
  return TCG_OK;
}

int grow_buffer(void** ptr, size_t* have, size_t want) {
  if (*have >= want) return TCG_OK;
  if (*ptr) {
    cudaError_t e = cudaFree(*ptr);  // synchronises: no queued kernel still uses it
    *ptr = nullptr;
    *have = 0;
    if (e != cudaSuccess) return record_cuda(e);
  }
  const size_t bytes = std::max(want, static_cast<size_t>(1) << 20);
  cudaError_t e = cudaMalloc(ptr, bytes);
  if (e != cudaSuccess) return record_cuda(e);
  *have = bytes;
  return TCG_OK;
}

int split_workspace(int dev, cudaStream_t s, size_t slot_bytes, float** slots) {
  std::lock_guard<std::mutex> lk(g_mu);
  SplitWorkspace& w = g_split_ws[std::make_pair(dev, s)];
  if (int rc = grow_buffer(&w.slots, &w.slot_bytes, slot_bytes)) return rc;
  *slots = static_cast<float*>(w.slots);
  return TCG_OK;
}

CUtensorMapDataType map_dtype(tcg_input t) {
  switch (t) {
    case TCG_IN_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case TCG_IN_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case TCG_IN_TF32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    // sixteen packed values per 16-byte block in shared memory (12 data
    // bytes, then padding)
    case TCG_IN_E3M2:
    case TCG_IN_E2M3: return CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
}

// Tensor map + descriptor constants for one operand tile of `rows` M/N rows
// and one ring stage of K (128 bytes).
int setup_operand(const void* ptr, tcg_input it, tcg_major major, int64_t mn, int64_t K, int64_t ld, int rows,
                  CUtensorMap* map, int* mn_major, int* boxes, int* box_mn, uint32_t* box_bytes, uint64_t* desc_hi,
                  uint32_t* kstep) {
  const int es = esize_of(it);
  const int bk = stage_k(it);  // K elements per stage
  const int mma_k = it == TCG_IN_TF32 ? 8 : is_fp4(it) ? 64 : is_mx(it) ? 32 : 16;
  const CUtensorMapDataType dt = map_dtype(it);
  if (major == TCG_K_MAJOR) {
    // rows enumerate M/N: one 128-byte swizzle row per M/N row, 8-row groups
    // 1024 bytes apart (SDO); the K step moves the start 32 bytes.
    *mn_major = 0;
    *boxes = 1;
    *box_mn = 0;
    *box_bytes = static_cast<uint32_t>(rows) * 128u;
    *desc_hi = sdesc_hi(16, 1024, SW_128B);
    // shared bytes of K per MMA issue: 32 (FP6 takes one padded byte per
    // element there; packed FP4 half a byte)
    *kstep = static_cast<uint32_t>(is_fp4(it) ? mma_k / 2 : mma_k * es);
    // the map's row stride is the global one (packed formats: ld * bits / 8);
    // packed FP4 is mapped as bytes (128-byte boxes of 256 values)
    const uint64_t inner = is_fp4(it) ? static_cast<uint64_t>(row_bytes(it, K)) : static_cast<uint64_t>(K);
    const uint32_t box_inner = is_fp4(it) ? 128u : static_cast<uint32_t>(bk);
    return make_map_2d(map, ptr, dt, 1, inner, static_cast<uint64_t>(mn), static_cast<uint64_t>(row_bytes(it, ld)),
                       box_inner, static_cast<uint32_t>(rows), CU_TENSOR_MAP_SWIZZLE_128B);
  }
  // MN-major: rows enumerate K; one 128-byte row holds 128/es M/N elements.
  *mn_major = 1;
  const int chunk = 128 / es;
  *box_mn = chunk;
  *boxes = (rows + chunk - 1) / chunk;
  *box_bytes = static_cast<uint32_t>(bk) * 128u;
  if (it == TCG_IN_TF32) {
    // "swizzle=4": four K rows of 128 bytes per SDO, LDO to the next 128-byte chunk
    *desc_hi = sdesc_hi(*box_bytes, 512, SW_128B_ATOM32);
    *kstep = static_cast<uint32_t>(mma_k / 4) * 512u;
  } else {
    *desc_hi = sdesc_hi(*box_bytes, 1024, SW_128B);
    *kstep = static_cast<uint32_t>(mma_k / 8) * 1024u;
  }
  return make_map_2d(map, ptr, dt, es, static_cast<uint64_t>(mn), static_cast<uint64_t>(K),
                     static_cast<uint64_t>(ld), static_cast<uint32_t>(chunk), static_cast<uint32_t>(bk),
                     it == TCG_IN_TF32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B);
}

int run_gemm(const tcg_gemm_args* args, cudaStream_t s) {
  load_timeout_env();
  t_last_launches = 0;
  t_plan = PlanRecord();
  if (!args) return TCG_ERR_INVALID;
  tcg_gemm_args a = *args;
  if (a.M < 0 || a.N < 0 || a.K < 0) return TCG_ERR_INVALID;
  if (a.in_type < TCG_IN_F16 || a.in_type > TCG_IN_NVF4) return TCG_ERR_INVALID;
  // the packed-FP4 kinds stage their scales with tcgen05.cp, from the MMA
  // thread or a copy thread (no tcgen05.st scale warps)
  if (is_fp4(a.in_type) && a.sf_staging == 1) return TCG_ERR_UNSUPPORTED;
  if (a.d_type < TCG_F32 || a.d_type > TCG_BF16 || a.acc_type < TCG_F32 || a.acc_type > TCG_BF16)
    return TCG_ERR_INVALID;
  if (a.acc_type == TCG_BF16) return TCG_ERR_UNSUPPORTED;
  if (a.acc_type == TCG_F16 && (a.in_type != TCG_IN_F16 || a.d_type != TCG_F16)) return TCG_ERR_UNSUPPORTED;
  if (a.cta_group < 0 || a.cta_group > 2 || a.raster_group < 0 || a.sf_staging < 0 || a.sf_staging > 3 ||
      a.split_k < -1 || a.epilogue < 0 || a.epilogue > 2)
    return TCG_ERR_INVALID;
  if (a.M > INT32_MAX / 2 || a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2) return TCG_ERR_UNSUPPORTED;
  if (a.M == 0 || a.N == 0) return TCG_OK;
  if (!a.D) return TCG_ERR_INVALID;
  if (a.ldd == 0) a.ldd = a.N;
  if (a.ldd < a.N) return TCG_ERR_INVALID;
  const int ds = dsize_of(a.d_type);
  if (reinterpret_cast<uintptr_t>(a.D) % ds) return TCG_ERR_ALIGNMENT;
  const bool scaled = is_mx(a.in_type);
  if (a.K > 0) {
    if (int rc = check_operand(a.A, a.a_major, a.M, a.K, &a.lda, a.in_type)) return rc;
    if (int rc = check_operand(a.B, a.b_major, a.N, a.K, &a.ldb, a.in_type)) return rc;
    if (scaled) {
      const bool plain = a.SFA || a.SFB;
      const bool img = a.SFA_img || a.SFB_img;
      if (plain == img) return TCG_ERR_INVALID;
      if (plain && (!a.SFA || !a.SFB)) return TCG_ERR_INVALID;
      if (img && (!a.SFA_img || !a.SFB_img)) return TCG_ERR_INVALID;
      if (img && ((reinterpret_cast<uintptr_t>(a.SFA_img) | reinterpret_cast<uintptr_t>(a.SFB_img)) % 16))
        return TCG_ERR_ALIGNMENT;
    } else if (a.SFA || a.SFB || a.SFA_img || a.SFB_img) {
      return TCG_ERR_INVALID;
    }
  }
  Plan plan;
  if (int rc = get_plan(a, &plan)) return rc;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  DeviceState* d = device_state(dev);

  if (a.K == 0) {
    const cudaError_t e = cudaMemset2DAsync(a.D, static_cast<size_t>(a.ldd) * ds, 0, static_cast<size_t>(a.N) * ds,
                                            static_cast<size_t>(a.M), s);
    if (e != cudaSuccess) return record_cuda(e);
    t_last_launches = 1;
    t_plan.valid = true;
    t_plan.k_zero = true;
    return TCG_OK;
  }

  bool d_trans = false;
  if (int rc = choose_plan(a, d->sms, &plan, &d_trans)) return rc;
  if (d_trans) {
    tcg_gemm_args t = a;
    t.M = a.N;
    t.N = a.M;
    t.A = a.B;
    t.a_major = a.b_major;
    t.lda = a.ldb;
    t.B = a.A;
    t.b_major = TCG_K_MAJOR;
    t.ldb = a.lda;
    a = t;
    if (int rc = get_plan(a, &plan)) return rc;
  }
  const KernelInfo& ki = plan.ki;
  const int cg = plan.cta_group;
  const int bn = ki.bn;
  GemmParams prm;
  std::memset(&prm, 0, sizeof prm);
  prm.M = static_cast<int>(a.M);
  prm.N = static_cast<int>(a.N);
  prm.K = static_cast<int>(a.K);
  prm.num_m_tiles = static_cast<int>(cdiv(a.M, 128 * cg));
  prm.num_n_tiles = static_cast<int>(cdiv(a.N, bn));
  prm.num_k_blocks = static_cast<int>(cdiv(a.K, stage_k(a.in_type)));
  // tile, unit and slot indices are 32-bit in the kernels
  if (static_cast<int64_t>(prm.num_m_tiles) * prm.num_n_tiles > INT32_MAX / 4) {
    t_last_error = "too many output tiles";
    return TCG_ERR_UNSUPPORTED;
  }
  prm.num_tiles = prm.num_m_tiles * prm.num_n_tiles;
  // M tiles per raster group: the rows of A whose tiles sweep N together
  // hold about 32 MiB (kept between 2048 and 8192 rows), so that they stay in
  // the L2 while B streams past.  Best group sizes measured (pairs, 8192^3
  // unless stated): bf16 8 (2048 rows), E4M3 16 (4096), E2M3 16-24, E2M1 32
  // (8192); bf16 K = 4096 16, K = 16384 8; E4M3 16384 x 8192 x 4096 16-32,
  // K = 16384 8; single CTAs bf16 8192^3 16 (2048 rows).
  const int64_t group_rows = std::min<int64_t>(8192, std::max<int64_t>(2048, (32LL << 20) / std::max<int64_t>(1, row_bytes(a.in_type, a.K))));
  prm.raster_group = a.raster_group > 0 ? a.raster_group : static_cast<int>(group_rows / (128 * cg));
  // a group of all M tiles is the widest there is (and keeps group x N tiles
  // within the tile count's 32-bit range)
  prm.raster_group = std::min(prm.raster_group, prm.num_m_tiles);
  // skinny single-CTA problems: the A box covers only the rows that exist
  const int a_rows = (cg == 1 && a.a_major == TCG_K_MAJOR && a.M < 128) ? static_cast<int>(cdiv(a.M, 8) * 8) : 128;
  if (int rc = setup_operand(a.A, a.in_type, a.a_major, a.M, a.K, a.lda, a_rows, &prm.tmap_a, &prm.a_mn_major,
                             &prm.a_boxes, &prm.a_box_mn, &prm.a_box_bytes, &prm.a_desc_hi, &prm.a_kstep))
    return rc;
  // bytes TMA writes per stage: 128 elements of K per row; the packed 6- and
  // 4-bit types write only their data bytes (96 / 64 per row) and skip the
  // padding of each 16-byte block
  prm.ab_tx_bytes = static_cast<uint32_t>((a_rows + bn / cg) * stage_row_tx(a.in_type) * cg);
  // 384-column pair tiles stage each CTA's 192 B rows as three 64-row boxes
  const int b_box_rows = bn > 256 ? 64 : bn / cg;
  if (int rc = setup_operand(a.B, a.in_type, a.b_major, a.N, a.K, a.ldb, b_box_rows, &prm.tmap_b, &prm.b_mn_major,
                             &prm.b_boxes, &prm.b_box_mn, &prm.b_box_bytes, &prm.b_desc_hi, &prm.b_kstep))
    return rc;
  const bool a_mn = a.a_major == TCG_MN_MAJOR, b_mn = a.b_major == TCG_MN_MAJOR;
  const int mma_n = std::min(bn, 256);  // a 384-column tile's first MMA; the kernel derives the second
  if (a.in_type == TCG_IN_TF32)
    prm.idesc = idesc_tf32(a_mn, b_mn, 128 * cg, bn);
  else if (is_fp4(a.in_type))
    prm.idesc = idesc_fp4(128 * cg, mma_n, a.in_type == TCG_IN_E2M1);
  else if (scaled)
    prm.idesc = idesc_mxf8(a_mn, b_mn, 128 * cg, mma_n, mx_format(a.in_type), mx_format(a.in_type));
  else
    prm.idesc = idesc_f16(a.in_type == TCG_IN_BF16, a.acc_type == TCG_F32, a_mn, b_mn, 128 * cg, bn);
  prm.D = a.D;
  prm.ldd = a.ldd;
  prm.d_type = a.d_type == TCG_F32 ? OUT_F32 : a.d_type == TCG_F16 ? OUT_F16 : OUT_BF16;
  prm.acc_f16 = a.acc_type == TCG_F16;
  prm.d_vec_ok = (reinterpret_cast<uintptr_t>(a.D) % 16 == 0) && ((a.ldd * ds) % 16 == 0);
  // Outputs leave through TMA tile stores (32 rows x 64 bytes: 32 columns of
  // 16-bit values, 16 of fp32) when the map's alignment rules hold (16-byte
  // base and row stride); otherwise per-thread row stores.  fp32 tiles
  // replace per-lane row stores, in which one warp store instruction touches
  // 32 rows.
  prm.d_tma = 0;
  prm.d_trans = d_trans ? 1 : 0;
  if (prm.d_vec_ok && !d_trans) {
    const CUtensorMapDataType dt = a.d_type == TCG_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : a.d_type == TCG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (int rc = make_map_2d(&prm.tmap_d, a.D, dt, ds, static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.M),
                             static_cast<uint64_t>(a.ldd), static_cast<uint32_t>(64 / ds), 32,
                             CU_TENSOR_MAP_SWIZZLE_64B))
      return rc;
    prm.d_tma = 1;
  }
  prm.epi_frag = a.epilogue == 2 ? 1 : 0;
  const bool frag_used = prm.epi_frag && prm.d_tma && a.d_type != TCG_F32 && a.acc_type == TCG_F32;
  prm.err = d->err;
  prm.timeout_ns = g_timeout_ns.load();
  prm.trace = t_trace_buf;
  prm.trace_ctas = t_trace_ctas;
  t_trace_buf = nullptr;
  t_trace_ctas = 0;
  // auto: the MMA warp copies the scales itself (fastest or tied for both
  // CTA groups once the issue loops are warp-uniform; no extra barriers)
  prm.sf_mode = a.sf_staging == 1   ? SF_BY_WARPS
                : a.sf_staging == 3 ? SF_BY_CP
                                    : SF_BY_MMA;

  int launches = 0;
  if (scaled) {
    const int sfa_tiles = static_cast<int>(cdiv(a.M, 128));
    const int chunks = static_cast<int>(cdiv(bn, 128));
    const int kch = scale_format(a.in_type).kch;  // 512-byte chunks per 128 rows per stage
    const int64_t ba = sf_image_bytes_fmt(a.in_type, a.M, a.K, 128);
    const int64_t bb = sf_image_bytes_fmt(a.in_type, a.N, a.K, bn);
    const uint8_t* sfa_img = a.SFA_img;
    const uint8_t* sfb_img = a.SFB_img;
    if (!sfa_img) {
      void* ws = nullptr;
      if (int rc = workspace(dev, s, static_cast<size_t>(ba + bb), &ws)) return rc;
      uint8_t* wa = static_cast<uint8_t*>(ws);
      uint8_t* wb = wa + ba;  // ba is a multiple of 512
      const cudaError_t e = launch_sf_prepare_pair(a.in_type, a.SFA, a.M, 128, wa, a.SFB, a.N, bn, wb, a.K, s);
      if (e != cudaSuccess) return record_cuda(e);
      launches += 1;
      sfa_img = wa;
      sfb_img = wb;
    }
    prm.sf_a_tiles = sfa_tiles;
    // one 512-byte chunk (128 words) per map row; a stage loads its kch
    // (SFA) or kch x chunks (SFB) consecutive rows in one box
    if (int rc = make_map_2d(&prm.tmap_sfa, sfa_img, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128,
                             static_cast<uint64_t>(ba / 512), 128, 128, static_cast<uint32_t>(kch),
                             CU_TENSOR_MAP_SWIZZLE_NONE))
      return rc;
    if (int rc = make_map_2d(&prm.tmap_sfb, sfb_img, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, 128,
                             static_cast<uint64_t>(bb / 512), 128, 128, static_cast<uint32_t>(kch * chunks),
                             CU_TENSOR_MAP_SWIZZLE_NONE))
      return rc;
  }

  int max_clusters = 0;
  if (int rc = max_clusters_for(d, ki, &max_clusters)) return rc;

  // Problems with few output tiles (skinny M or N) leave most SMs idle: by
  // default they run stream-K (each cluster takes an equal contiguous share
  // of the (tile, k block) iterations; tiles cut between clusters meet in an
  // fp32 workspace and a second kernel).  That costs a few microseconds and a
  // second epilogue per cluster, so it is used only when the tiles fill at
  // most a quarter of the clusters and the idle share times the K blocks is
  // at least 60 (measured with 128 x 256 tiles: 16 x 8192 x 8192 and
  // 64 x 4096 x 16384 gain; 128 x 16384 x 4096, 512 x 4096 x 4096 and
  // 2048^2 x 2048..8192 lose).  The
  // narrow (32-column) and skinny (64-column) tiles carry so little work per
  // tile that half the clusters suffice (16 x 4096 x 16384: 41 us stream-K vs
  // 60 us one pass; 8192 x 16 x 8192: 40 vs 58 us).
  // split_k >= 2 asks for a fixed split of every tile instead.  f16
  // accumulation keeps its single-pass path.
  int split = 1;
  bool stream_k = false;
  if (a.acc_type != TCG_F16) {
    if (a.split_k > 1)
      split = static_cast<int>(std::min<int64_t>({a.split_k, prm.num_k_blocks,
                                                  std::max<int64_t>(1, (INT32_MAX / 4) / prm.num_tiles)}));
    else if (a.split_k == -1)
      stream_k = true;
    else if (a.split_k == 0 && (bn <= 64 ? 2 : 4) * static_cast<int64_t>(prm.num_tiles) <= max_clusters &&
             static_cast<int64_t>(max_clusters - prm.num_tiles) * prm.num_k_blocks >= 60LL * max_clusters)
      stream_k = true;
  }
  prm.split = split;
  prm.stream_k = stream_k ? 1 : 0;
  prm.num_units = prm.num_tiles * split;
  const int64_t iterations = static_cast<int64_t>(prm.num_tiles) * prm.num_k_blocks;
  const int clusters = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(stream_k ? iterations : prm.num_units, max_clusters)));
  if (split > 1 || stream_k) {
    // partial-tile slots: under stream-K two per cluster (the two ends of its
    // range), under split-K one per unit; each CG x min(128, M) x BN fp32
    prm.w_rows = static_cast<int>(std::min<int64_t>(128, a.M));
    const int64_t slots = stream_k ? 2 * static_cast<int64_t>(clusters) : static_cast<int64_t>(prm.num_units);
    const int64_t wbytes = slots * cg * prm.w_rows * bn * 4;
    if (int rc = split_workspace(dev, s, static_cast<size_t>(wbytes), &prm.w)) return rc;
    prm.bn = bn;
    if (int rc = make_map_3d(&prm.tmap_w, prm.w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, static_cast<uint64_t>(bn),
                             static_cast<uint64_t>(prm.w_rows), static_cast<uint64_t>(slots * cg), 16, 32,
                             CU_TENSOR_MAP_SWIZZLE_64B))
      return rc;
  }
  if (int rc = launch_gemm(ki, prm, clusters, s)) return rc;
  launches += 1;
  if (split > 1 || stream_k) {
    const cudaError_t e = launch_splitk_reduce(prm, cg, clusters, s);
    if (e != cudaSuccess) return record_cuda(e);
    launches += 1;
  }
  t_last_launches = launches;
  t_plan.valid = true;
  t_plan.cg = cg;
  t_plan.bn = bn;
  t_plan.clusters = clusters;
  t_plan.split = split;
  t_plan.swapped = d_trans;
  t_plan.stream_k = stream_k;
  t_plan.frag = frag_used;
  return TCG_OK;
}

}  // namespace

int record_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TCG_OK;
  t_last_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
  return TCG_ERR_CUDA;
}

int current_device_checked(int* dev) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) {
    record_cuda(e);
    cudaGetLastError();
    return TCG_ERR_NO_DEVICE;
  }
  DeviceState* st = device_state(d);
  if (!st || !st->usable) {
    t_last_error = "current device is not an sm_103 GPU";
    return TCG_ERR_NO_DEVICE;
  }
  // The tensor maps are encoded with a driver call, which needs a context
  // current on this thread; a host thread that has made no runtime call that
  // binds one yet gets the device's primary context (the one the runtime
  // itself would use).  A context the caller made current is left alone.
  std::call_once(g_ctx_get_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    else
      cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  if (g_ctx_get && g_ctx_get(&ctx) == CUDA_SUCCESS && ctx == nullptr) {
    e = cudaSetDevice(d);
    if (e != cudaSuccess) return record_cuda(e);
  }
  *dev = d;
  return TCG_OK;
}

unsigned long long* device_error_word(int dev) {
  DeviceState* st = device_state(dev);
  return st ? st->err : nullptr;
}

uint64_t wait_timeout_ns() {
  load_timeout_env();
  return g_timeout_ns.load();
}

void set_launch_count(int n) { t_last_launches = n; }

void set_error_message(const char* msg) { t_last_error = msg ? msg : ""; }

}  // namespace tcg

using namespace tcg;

namespace {

int named_gemm(tcg_input in, int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda,
               const void* B, tcg_major b_major, int64_t ldb, const uint8_t* SFA, const uint8_t* SFB, void* D,
               tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type, void* stream) {
  tcg_gemm_args a;
  std::memset(&a, 0, sizeof a);
  a.M = M;
  a.N = N;
  a.K = K;
  a.in_type = in;
  a.A = A;
  a.a_major = a_major;
  a.lda = lda;
  a.B = B;
  a.b_major = b_major;
  a.ldb = ldb;
  a.SFA = SFA;
  a.SFB = SFB;
  a.D = D;
  a.d_type = d_type;
  a.ldd = ldd;
  a.acc_type = acc_type;
  return run_gemm(&a, reinterpret_cast<cudaStream_t>(stream));
}

// E = round(A . B1) . B2 through one kernel (gemm_chain.cu).
int run_chain(tcg_input in, int64_t M, int64_t N1, int64_t N2, int64_t K, const void* A, int64_t lda,
              const void* B1, int64_t ldb1, const void* B2, int64_t ldb2, void* E, tcg_dtype e_type, int64_t lde,
              cudaStream_t s) {
  t_last_launches = 0;
  t_plan = PlanRecord();
  if (in != TCG_IN_F16 && in != TCG_IN_BF16) return TCG_ERR_INVALID;
  if (M < 0 || N2 < 0 || K < 0 || N1 < 16 || N1 > 256 || N1 % 16) return TCG_ERR_INVALID;
  if (e_type < TCG_F32 || e_type > TCG_BF16) return TCG_ERR_INVALID;
  if (M > INT32_MAX / 2 || N2 > INT32_MAX / 2 || K > INT32_MAX / 2) return TCG_ERR_UNSUPPORTED;
  if (M == 0 || N2 == 0) return TCG_OK;
  if (!E) return TCG_ERR_INVALID;
  if (lde == 0) lde = N2;
  if (lde < N2) return TCG_ERR_INVALID;
  const int es = dsize_of(e_type);
  // E leaves through TMA tile stores: 16-byte base and row stride
  if (reinterpret_cast<uintptr_t>(E) % 16 || (lde * es) % 16) return TCG_ERR_ALIGNMENT;
  if (K > 0) {
    if (int rc = check_operand(A, TCG_K_MAJOR, M, K, &lda, in)) return rc;
    if (int rc = check_operand(B1, TCG_K_MAJOR, N1, K, &ldb1, in)) return rc;
  }
  if (int rc = check_operand(B2, TCG_K_MAJOR, N2, N1, &ldb2, in)) return rc;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  DeviceState* d = device_state(dev);
  if (K == 0) {  // C = 0, so E = 0
    const cudaError_t e = cudaMemset2DAsync(E, static_cast<size_t>(lde) * es, 0, static_cast<size_t>(N2) * es,
                                            static_cast<size_t>(M), s);
    if (e != cudaSuccess) return record_cuda(e);
    t_last_launches = 1;
    return TCG_OK;
  }
  const CUtensorMapDataType dt = in == TCG_IN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  // Pairs of CTAs on neighbouring row tiles share every B1 / B2 tile: each
  // loads half of its rows and multicasts them to both, so an SM pulls half
  // of the B bytes from L2.  Measured on 38912-row problems: 8 % faster at
  // N1 = 256, even at N1 = 128, 2 % slower at N1 = 64 (little B traffic to
  // save); and 5 % slower on 8 row tiles, where the units are short.
  // Clusters of four were slower everywhere but at 8192 x 256 x 8192 x 8192.
  const int64_t m_tiles = cdiv(M, 128);
  const int cs = m_tiles >= 16 && N1 >= 128 ? 2 : 1;
  const KernelInfo ki = kinfo_chain(cs);
  int clusters = 0;
  if (int rc = max_clusters_for(d, ki, &clusters)) return rc;
  ChainParams p;
  std::memset(&p, 0, sizeof p);
  if (int rc = make_map_2d(&p.tmap_a, A, dt, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(lda), 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
    return rc;
  if (int rc = make_map_2d(&p.tmap_b1, B1, dt, 2, static_cast<uint64_t>(K), static_cast<uint64_t>(N1),
                           static_cast<uint64_t>(ldb1), 64, static_cast<uint32_t>(N1 / cs), CU_TENSOR_MAP_SWIZZLE_128B))
    return rc;
  if (int rc = make_map_2d(&p.tmap_b2, B2, dt, 2, static_cast<uint64_t>(N1), static_cast<uint64_t>(N2),
                           static_cast<uint64_t>(ldb2), 64, static_cast<uint32_t>(CHAIN_BN2 / cs),
                           CU_TENSOR_MAP_SWIZZLE_128B))
    return rc;
  const CUtensorMapDataType et = e_type == TCG_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : e_type == TCG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  if (int rc = make_map_2d(&p.tmap_e, E, et, es, static_cast<uint64_t>(N2), static_cast<uint64_t>(M),
                           static_cast<uint64_t>(lde), static_cast<uint32_t>(64 / es), 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return rc;
  p.M = static_cast<int>(M);
  p.N1 = static_cast<int>(N1);
  p.N2 = static_cast<int>(N2);
  p.K = static_cast<int>(K);
  p.m_tiles = static_cast<int>(m_tiles);
  p.m_blocks = static_cast<int>(cdiv(m_tiles, cs));
  p.n2_tiles = static_cast<int>(cdiv(N2, CHAIN_BN2));
  // Fewer row blocks than clusters: split the E tiles into groups (each
  // group's unit recomputes its rows of C) so that about every SM has a unit.
  const int64_t groups_wanted = std::max<int64_t>(1, std::min<int64_t>(p.n2_tiles, clusters / p.m_blocks));
  p.tiles_per_group = static_cast<int>(cdiv(p.n2_tiles, groups_wanted));
  const int64_t groups = cdiv(p.n2_tiles, p.tiles_per_group);
  if (static_cast<int64_t>(p.m_blocks) * groups > INT32_MAX / 2) return TCG_ERR_UNSUPPORTED;
  p.num_units = static_cast<int>(p.m_blocks * groups);
  p.k1_blocks = static_cast<int>(cdiv(K, 64));
  p.k2_blocks = static_cast<int>(cdiv(N1, 128));
  p.k2_steps = static_cast<int>(N1 / 16);
  const bool bf = in == TCG_IN_BF16;
  p.idesc1 = idesc_f16(bf, true, false, false, 128, static_cast<int>(N1));
  p.idesc2 = idesc_f16(bf, true, false, false, 128, CHAIN_BN2);
  p.in_bf16 = bf ? 1 : 0;
  p.e_type = e_type == TCG_F32 ? OUT_F32 : e_type == TCG_F16 ? OUT_F16 : OUT_BF16;
  p.err = d->err;
  p.timeout_ns = g_timeout_ns.load();
  p.trace = t_trace_buf;
  p.trace_ctas = t_trace_ctas;
  t_trace_buf = nullptr;
  t_trace_ctas = 0;
  const int grid = cs * static_cast<int>(std::min<int64_t>(p.num_units, clusters));
  const cudaError_t e = launch_chain(p, cs, grid, s);
  if (e != cudaSuccess) return record_cuda(e);
  t_last_launches = 1;
  t_plan.valid = true;
  t_plan.k_zero = false;
  t_plan.cg = 1;
  t_plan.mc = cs;
  t_plan.bn = CHAIN_BN2;
  t_plan.clusters = grid / cs;
  t_plan.split = 1;
  t_plan.swapped = false;
  t_plan.stream_k = false;
  t_plan.frag = false;
  return TCG_OK;
}

}  // namespace

extern "C" {

int tcg_gemm_chain(tcg_input in_type, int64_t M, int64_t N1, int64_t N2, int64_t K, const void* A, int64_t lda,
                   const void* B1, int64_t ldb1, const void* B2, int64_t ldb2, void* E, tcg_dtype e_type, int64_t lde,
                   void* stream) {
  return run_chain(in_type, M, N1, N2, K, A, lda, B1, ldb1, B2, ldb2, E, e_type, lde,
                   reinterpret_cast<cudaStream_t>(stream));
}

int tcg_gemm(const tcg_gemm_args* args, void* stream) {
  return run_gemm(args, reinterpret_cast<cudaStream_t>(stream));
}

int tcg_gemm_f16(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda, const void* B,
                 tcg_major b_major, int64_t ldb, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                 void* stream) {
  return named_gemm(TCG_IN_F16, M, N, K, A, a_major, lda, B, b_major, ldb, nullptr, nullptr, D, d_type, ldd, acc_type,
                    stream);
}

int tcg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda, const void* B,
                  tcg_major b_major, int64_t ldb, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                  void* stream) {
  return named_gemm(TCG_IN_BF16, M, N, K, A, a_major, lda, B, b_major, ldb, nullptr, nullptr, D, d_type, ldd,
                    acc_type, stream);
}

int tcg_gemm_tf32(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda, const void* B,
                  tcg_major b_major, int64_t ldb, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                  void* stream) {
  return named_gemm(TCG_IN_TF32, M, N, K, A, a_major, lda, B, b_major, ldb, nullptr, nullptr, D, d_type, ldd,
                    acc_type, stream);
}

int tcg_gemm_mxf8_blockscaled(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb, const uint8_t* SFA,
                              const uint8_t* SFB, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                              void* stream) {
  if (K > 0 && (!SFA || !SFB)) return TCG_ERR_INVALID;
  return named_gemm(TCG_IN_E4M3, M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type,
                    stream);
}

int tcg_gemm_mxf6_blockscaled(tcg_input fmt, int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major,
                              int64_t lda, const void* B, tcg_major b_major, int64_t ldb, const uint8_t* SFA,
                              const uint8_t* SFB, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                              void* stream) {
  if (fmt != TCG_IN_E3M2 && fmt != TCG_IN_E2M3) return TCG_ERR_INVALID;
  if (K > 0 && (!SFA || !SFB)) return TCG_ERR_INVALID;
  return named_gemm(fmt, M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type, stream);
}

int tcg_gemm_mxf4_blockscaled(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb, const uint8_t* SFA,
                              const uint8_t* SFB, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                              void* stream) {
  if (K > 0 && (!SFA || !SFB)) return TCG_ERR_INVALID;
  return named_gemm(TCG_IN_E2M1, M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type,
                    stream);
}

int tcg_gemm_nvf4_blockscaled(int64_t M, int64_t N, int64_t K, const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb, const uint8_t* SFA,
                              const uint8_t* SFB, void* D, tcg_dtype d_type, int64_t ldd, tcg_dtype acc_type,
                              void* stream) {
  if (K > 0 && (!SFA || !SFB)) return TCG_ERR_INVALID;
  return named_gemm(TCG_IN_NVF4, M, N, K, A, a_major, lda, B, b_major, ldb, SFA, SFB, D, d_type, ldd, acc_type,
                    stream);
}

int64_t tcg_scale_image_bytes(tcg_input fmt, int64_t rows, int64_t K, int tile_rows) {
  if (rows < 0 || K < 0 || tile_rows <= 0 || !is_mx(fmt)) return -1;
  return sf_image_bytes_fmt(fmt, rows, K, tile_rows);
}

int tcg_prepare_scales_ab(tcg_input fmt, const uint8_t* SFA, int64_t M, uint8_t* SFA_img, const uint8_t* SFB,
                          int64_t N, int tile_n, uint8_t* SFB_img, int64_t K, void* stream) {
  if (!is_mx(fmt) || M < 0 || N < 0 || K < 0 || tile_n <= 0 || tile_n > 65536) return TCG_ERR_INVALID;
  if (K == 0 || (M == 0 && N == 0)) return TCG_OK;
  if ((M > 0 && (!SFA || !SFA_img)) || (N > 0 && (!SFB || !SFB_img))) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaError_t e = launch_sf_prepare_pair(fmt, M > 0 ? SFA : nullptr, M, 128, SFA_img, N > 0 ? SFB : nullptr,
                                               N, tile_n, SFB_img, K, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e);
  set_launch_count(1);
  return TCG_OK;
}

int64_t tcg_mxf8_scale_image_bytes(int64_t rows, int64_t K, int tile_rows) {
  return tcg_scale_image_bytes(TCG_IN_E4M3, rows, K, tile_rows);
}

int tcg_tile_n(tcg_input fmt, int64_t M, int64_t N, int64_t K, tcg_major b_major, int cta_group) {
  if (!is_mx(fmt)) return TCG_ERR_INVALID;
  tcg_gemm_args a;
  std::memset(&a, 0, sizeof a);
  a.M = M;
  a.N = N;
  a.K = K;
  a.in_type = fmt;
  a.b_major = b_major;
  a.cta_group = cta_group;
  Plan p;
  if (int rc = get_plan(a, &p)) return rc;
  return p.ki.bn;
}

int tcg_mxf8_tile_n(int64_t M, int64_t N, int64_t K, tcg_major b_major, int cta_group) {
  return tcg_tile_n(TCG_IN_E4M3, M, N, K, b_major, cta_group);
}

int tcg_mxf8_prepare_scales(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows, uint8_t* img, void* stream) {
  if (rows < 0 || K < 0 || tile_rows <= 0 || tile_rows > 65536) return TCG_ERR_INVALID;
  if (rows == 0 || K == 0) return TCG_OK;
  if (!sf || !img) return TCG_ERR_INVALID;
  int dev;
  if (int rc = current_device_checked(&dev)) return rc;
  const cudaError_t e =
      launch_sf_prepare(TCG_IN_E4M3, sf, rows, K, tile_rows, img, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e);
  set_launch_count(1);
  return TCG_OK;
}

int tcg_mxf8_prepare_scales_ab(const uint8_t* SFA, int64_t M, uint8_t* SFA_img, const uint8_t* SFB, int64_t N,
                               int tile_n, uint8_t* SFB_img, int64_t K, void* stream) {
  return tcg_prepare_scales_ab(TCG_IN_E4M3, SFA, M, SFA_img, SFB, N, tile_n, SFB_img, K, stream);
}

int tcg_check(void* stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e);
  DeviceState* st = device_state(dev);
  if (!st || !st->err) return TCG_OK;
  unsigned long long w = 0;
  e = cudaMemcpy(&w, st->err, sizeof w, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return record_cuda(e);
  if (w == 0) return TCG_OK;
  e = cudaMemset(st->err, 0, sizeof w);
  if (e != cudaSuccess) return record_cuda(e);
  char buf[128];
  std::snprintf(buf, sizeof buf, "kernel wait timed out (site %llu, block %llu)", (w >> 8) & 0xFF, (w >> 16) & 0xFFFFFFFF);
  t_last_error = buf;
  return (w & 0xFF) == 1 ? TCG_ERR_TIMEOUT : TCG_ERR_CUDA;
}

void tcg_set_wait_timeout_ns(uint64_t ns) {
  load_timeout_env();
  g_timeout_ns.store(ns < 1000 ? 1000 : ns);
}

const char* tcg_status_string(int status) {
  switch (status) {
    case TCG_OK: return "ok";
    case TCG_ERR_INVALID: return "invalid argument";
    case TCG_ERR_ALIGNMENT: return "misaligned pointer or leading dimension (TMA needs 16-byte alignment)";
    case TCG_ERR_UNSUPPORTED: return "unsupported combination";
    case TCG_ERR_CUDA: return "CUDA error";
    case TCG_ERR_TIMEOUT: return "kernel wait timed out";
    case TCG_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

const char* tcg_last_error_string(void) { return t_last_error.c_str(); }

int tcg_last_launch_count(void) { return t_last_launches; }

const char* tcg_last_plan_string(void) {
  const PlanRecord& p = t_plan;
  if (!p.valid) {
    t_last_plan.clear();
  } else if (p.k_zero) {
    t_last_plan = "K = 0: D zeroed";
  } else {
    char buf[200];
    std::snprintf(buf, sizeof buf, "cta_group %d, tile %dx%d%s, %d clusters%s, %s%s%s", p.cg, 128 * p.cg, p.bn,
                  p.swapped ? " (operands swapped, D stored transposed)" : "", p.clusters,
                  p.mc > 1 ? (" of " + std::to_string(p.mc) + " sharing B by multicast").c_str() : "",
                  p.stream_k ? "stream-K" : p.split > 1 ? "split-K " : "one pass per tile",
                  p.split > 1 ? std::to_string(p.split).c_str() : "",
                  p.frag ? ", 16x256b + stmatrix epilogue" : "");
    t_last_plan = buf;
  }
  return t_last_plan.c_str();
}

int tcg_trace_next(unsigned long long* buf, int max_ctas) {
  if ((buf == nullptr) != (max_ctas == 0) || max_ctas < 0) return TCG_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(buf) % 8) return TCG_ERR_ALIGNMENT;
  t_trace_buf = buf;
  t_trace_ctas = max_ctas;
  return TCG_OK;
}

}  // extern "C"
