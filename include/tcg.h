/*
 * tcg.h -- C ABI of the GB300 (sm_103a) tcgen05 swizzled GEMM library.
 *
 * The operation is the dense contraction that the Apache TVM TIRx
 * "tcgen05.mma" page defines ("Operands and repeat axes": D, A, B with A and B
 * in shared memory, D an fp32/fp16 accumulator in tensor memory), tiled over
 * a whole matrix:
 *
 *     D[m, n] = sum_k A[m, k] * B[k, n]                 (gemm_f16/bf16/tf32)
 *     D[m, n] = sum_k (SFA (.) A)[m, k] * (SFB (.) B)[k, n]   (block scaled,
 *               "Weight-stationary and block scaling": one e8m0 scale per 32
 *               K elements per row of A and per column of B)
 *
 * Operand majorness follows the page's descriptor contract ("Shared
 * descriptors are byte-stride contracts": K-major rows enumerate M/N,
 * MN-major rows enumerate K):
 *     A, TCG_K_MAJOR : M x K row-major, element (m,k) at A[m*lda + k]
 *     A, TCG_MN_MAJOR: K x M row-major, element (m,k) at A[k*lda + m]
 *     B, TCG_K_MAJOR : N x K row-major, element (k,n) at B[n*ldb + k]
 *     B, TCG_MN_MAJOR: K x N row-major, element (k,n) at B[k*ldb + n]
 *     D              : M x N row-major, element (m,n) at D[m*ldd + n]
 * A leading dimension of 0 means "packed" (K, M, N or N as appropriate).
 *
 * Ownership: every pointer is caller-owned DEVICE memory (except where a
 * function says host) that must stay valid until the work queued on `stream`
 * has finished.  D must not overlap A, B or the scale arrays (tiles of D are
 * written while other tiles still read the operands).  All calls are asynchronous on `stream` (a cudaStream_t; 0 is
 * the legacy default stream) and never synchronise the host, except
 * tcg_check().  The block-scaled GEMM with plain scale arrays, and split-K
 * (see tcg_gemm_args::split_k; automatic for problems with few output tiles),
 * use library-owned device workspaces per (device, stream), allocated on
 * first use and grown when needed (growing frees the old one, which waits for
 * the device); nothing else allocates device memory.  Calls on different
 * streams use different workspaces and may run concurrently.  A call may be
 * captured into a CUDA graph once an earlier call on the same stream has
 * allocated a workspace at least as large (a workspace that would have to
 * grow during capture fails the call with TCG_ERR_CUDA); the graph reuses
 * that stream's workspace, so its replays must be ordered with that stream's
 * other split-K / block-scaled work.
 *
 * Errors: every function returns TCG_OK (0) or a negative tcg_status.
 * Argument errors are detected on the host before anything is queued.
 * Device-side failures (a bounded wait in a kernel that ran out, see
 * tcg_set_wait_timeout_ns) are recorded in a per-device error word and
 * reported by the next tcg_check().
 */
#ifndef TCG_H_
#define TCG_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TCG_OK = 0,
  TCG_ERR_INVALID = -1,     /* null pointer, negative size, bad enum, ld too small */
  TCG_ERR_ALIGNMENT = -2,   /* TMA needs 16-byte aligned bases and row strides */
  TCG_ERR_UNSUPPORTED = -3, /* valid request this library does not implement */
  TCG_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed (see tcg_last_error_string) */
  TCG_ERR_TIMEOUT = -5,     /* a kernel's bounded mbarrier wait ran out (from tcg_check) */
  TCG_ERR_NO_DEVICE = -6    /* no usable sm_103 device */
} tcg_status;

typedef enum { TCG_K_MAJOR = 0, TCG_MN_MAJOR = 1 } tcg_major;

/* Accumulator / output element types. */
typedef enum { TCG_F32 = 0, TCG_F16 = 1, TCG_BF16 = 2 } tcg_dtype;

/* Operand storage types (generic entry point).  The block-scaled formats
 * ("tcgen05.mma" page, "Weight-stationary and block scaling": ".kind and
 * .scale_vec::1X/2X/4X"):
 *   E4M3, E5M2, E3M2, E2M3  kind::mxf8f6f4.block_scale.scale_vec::1X, one e8m0
 *                           scale per 32 K elements;
 *   E2M1 (MXFP4)            kind::mxf4.block_scale.scale_vec::2X, e8m0 per 32;
 *   NVF4 (NVFP4)            E2M1 elements, kind::mxf4nvf4.block_scale.
 *                           scale_vec::4X, one unsigned E4M3 scale per 16.
 * E3M2, E2M3 and the FP4 formats are stored packed: element i of the array
 * (i = row * ld + column, ld counted in elements) in bits [b*i, b*(i+1)) of
 * the array read as one little-endian bit string (b = 6 or 4; an FP4 byte
 * holds element 2j in its low nibble).  In shared memory the FP6 values sit
 * sixteen to a 16-byte block, data first and padding after -- the layout of
 * the "tcgen05.cp" page's "Native FP4/FP6 decompression" sources -- so a
 * 128-byte row holds 128 of them; FP4 stays packed, 256 to a row. */
typedef enum {
  TCG_IN_F16 = 0,   /* IEEE binary16, MMA kind::f16 */
  TCG_IN_BF16 = 1,  /* bfloat16, kind::f16 */
  TCG_IN_TF32 = 2,  /* float32 storage read as TF32, kind::tf32 */
  TCG_IN_E4M3 = 3,  /* OCP E4M3FN (FP8) */
  TCG_IN_E5M2 = 4,  /* OCP E5M2 (FP8) */
  TCG_IN_E3M2 = 5,  /* OCP MX E3M2 (FP6), packed */
  TCG_IN_E2M3 = 6,  /* OCP MX E2M3 (FP6), packed */
  TCG_IN_E2M1 = 7,  /* OCP MX E2M1 (FP4), packed, e8m0 scales per 32 */
  TCG_IN_NVF4 = 8   /* E2M1 (FP4), packed, unsigned E4M3 scales per 16 (NVFP4) */
} tcg_input;

/* ---------------------------------------------------------------------------
 * The four GEMMs.  M, N, K >= 0 (M == 0 or N == 0: no-op; K == 0: D = 0).
 * acc_type: TCG_F32, or TCG_F16 for gemm_f16 only (fp16 accumulation in TMEM,
 * output then must be TCG_F16).  d_type: TCG_F32, TCG_F16 or TCG_BF16.
 * Alignment: A, B base addresses and lda*sizeof, ldb*sizeof must be multiples
 * of 16 bytes (TMA); D must be at least 2-byte aligned (4 for F32).
 * ------------------------------------------------------------------------- */
int tcg_gemm_f16(int64_t M, int64_t N, int64_t K,
                 const void* A, tcg_major a_major, int64_t lda,
                 const void* B, tcg_major b_major, int64_t ldb,
                 void* D, tcg_dtype d_type, int64_t ldd,
                 tcg_dtype acc_type, void* stream);

int tcg_gemm_bf16(int64_t M, int64_t N, int64_t K,
                  const void* A, tcg_major a_major, int64_t lda,
                  const void* B, tcg_major b_major, int64_t ldb,
                  void* D, tcg_dtype d_type, int64_t ldd,
                  tcg_dtype acc_type, void* stream);

/* A and B are float32 storage; the tensor cores read them as TF32
 * ("tcgen05.mma" page, "Operands": the tf32 format is given explicitly for
 * float32 storage).  MN-major TF32 uses the 128-byte-span / 32-byte-atom
 * swizzle ("swizzle=4" section). */
int tcg_gemm_tf32(int64_t M, int64_t N, int64_t K,
                  const void* A, tcg_major a_major, int64_t lda,
                  const void* B, tcg_major b_major, int64_t ldb,
                  void* D, tcg_dtype d_type, int64_t ldd,
                  tcg_dtype acc_type, void* stream);

/* MXFP8: A, B are E4M3FN bytes; SFA is a plain row-major [M][ceil(K/32)]
 * e8m0 array, SFB [N][ceil(K/32)] (one scale per 32 K elements per row of A
 * and per column of B).  Scales are rearranged on the device into the
 * tcgen05.cp-ready image (tcg_mxf8_prepare_scales) in a library workspace,
 * then staged into TMEM with tcgen05.cp .32x128b.warpx4 ("tcgen05.cp" page,
 * shape table; "tcgen05.mma" page, block-scale placement).  acc_type must be
 * TCG_F32.  Uses the per-(device, stream) workspace described above: calls on
 * one stream are ordered; calls on different streams use different buffers. */
int tcg_gemm_mxf8_blockscaled(int64_t M, int64_t N, int64_t K,
                              const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb,
                              const uint8_t* SFA, const uint8_t* SFB,
                              void* D, tcg_dtype d_type, int64_t ldd,
                              tcg_dtype acc_type, void* stream);

/* Block-scaled FP6 GEMM (fmt TCG_IN_E3M2 or TCG_IN_E2M3): the MXFP8 operation
 * with 6-bit elements on the same MMA kind (kind::mxf8f6f4, the format in the
 * instruction descriptor) and scale layout (SFA [M][ceil(K/32)], SFB
 * [N][ceil(K/32)] e8m0).  A and B are packed (see tcg_input), K-major only
 * (TCG_ERR_UNSUPPORTED otherwise), lda / ldb count elements.  The tensor-map
 * rules of the padded element type apply: K a multiple of 128, A and B
 * 32-byte aligned, row strides (ld * 6 / 8 bytes) multiples of 32 bytes (else
 * TCG_ERR_ALIGNMENT).  acc_type must be TCG_F32.
 *
 * Block-scaled FP4 GEMMs: MXFP4 (E2M1, e8m0 scales [rows][ceil(K/32)],
 * kind::mxf4.block_scale.scale_vec::2X) and NVFP4 (E2M1, unsigned E4M3 scales
 * [rows][ceil(K/16)], kind::mxf4nvf4.block_scale.scale_vec::4X).  A and B are
 * packed two values per byte, K-major only; K and lda / ldb (in elements)
 * multiples of 32, A and B 16-byte aligned (else TCG_ERR_ALIGNMENT).  The
 * values stay packed in shared memory, 256 of K per 128-byte row and K = 64
 * per MMA.  acc_type must be TCG_F32. */
int tcg_gemm_mxf6_blockscaled(tcg_input fmt, int64_t M, int64_t N, int64_t K,
                              const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb,
                              const uint8_t* SFA, const uint8_t* SFB,
                              void* D, tcg_dtype d_type, int64_t ldd,
                              tcg_dtype acc_type, void* stream);

int tcg_gemm_mxf4_blockscaled(int64_t M, int64_t N, int64_t K,
                              const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb,
                              const uint8_t* SFA, const uint8_t* SFB,
                              void* D, tcg_dtype d_type, int64_t ldd,
                              tcg_dtype acc_type, void* stream);

int tcg_gemm_nvf4_blockscaled(int64_t M, int64_t N, int64_t K,
                              const void* A, tcg_major a_major, int64_t lda,
                              const void* B, tcg_major b_major, int64_t ldb,
                              const uint8_t* SFA, const uint8_t* SFB,
                              void* D, tcg_dtype d_type, int64_t ldd,
                              tcg_dtype acc_type, void* stream);

/* Same operation and arguments as tcg_gemm_mxf8_blockscaled, for callers that
 * must not allocate device memory (for example a framework whose caching
 * allocator owns all device memory, or code that cannot afford the
 * device-wide wait of a cudaFree when a workspace grows).  No counterpart on
 * the source pages: it only changes where the scale-factor images live.
 * They are built in one fixed 16 MiB device array of the library (held by
 * every GPU that loads the library until exit) instead of the per-stream
 * workspace; problems whose two images need more return TCG_ERR_UNSUPPORTED.
 * Every argument is checked before anything is queued, so a call that returns
 * an error has not touched the array.  All calls on a device share it (each
 * call rewrites what it reads, so nothing needs clearing); calls whose GPU
 * work overlaps race on it and must be ordered.  The first call on a device
 * looks up the array's address with that device current: make it before any
 * stream capture.  Allocates nothing (no cudaMalloc/cudaFree). */
int tcg_gemm_mxf8_blockscaled_noalloc(int64_t M, int64_t N, int64_t K,
                                      const void* A, tcg_major a_major, int64_t lda,
                                      const void* B, tcg_major b_major, int64_t ldb,
                                      const uint8_t* SFA, const uint8_t* SFB,
                                      void* D, tcg_dtype d_type, int64_t ldd,
                                      tcg_dtype acc_type, void* stream);

/* ---------------------------------------------------------------------------
 * Generic entry point: every knob of the four calls above plus the CTA-group
 * and tile choices (0 = let the library choose).
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t M, N, K;
  tcg_input in_type;
  const void* A; tcg_major a_major; int64_t lda;
  const void* B; tcg_major b_major; int64_t ldb;
  /* block scaling (TCG_IN_E4M3 .. TCG_IN_E2M1): either plain scales ... */
  const uint8_t* SFA; const uint8_t* SFB;
  /* ... or images already built by tcg_mxf8_prepare_scales (then SFA/SFB must
   * be NULL).  The images must have been prepared for the same M/N/K and the
   * tile_n this call resolves to (tcg_tile_n). */
  const uint8_t* SFA_img; const uint8_t* SFB_img;
  void* D; tcg_dtype d_type; int64_t ldd;
  tcg_dtype acc_type;
  int cta_group;     /* 0 auto (pairs once M > 128 and N >= 1024), 1 (one CTA per
                        128xN tile), 2 (CTA pair, 256xN) */
  int raster_group;  /* 0 auto; tiles are visited in groups of this many M tiles */
  int sf_staging;    /* block scaling, who stages the scales into TMEM:
                        0 = auto (2),
                        1 = four scale warps per CTA with tcgen05.st
                            (8- and 6-bit formats; packed FP4:
                            TCG_ERR_UNSUPPORTED),
                        2 = the MMA thread with tcgen05.cp .32x128b.warpx4
                            ("tcgen05.cp" page) before its MMAs,
                        3 = a dedicated thread with tcgen05.cp + commit */
  int split_k;       /* K decomposition: 0 = auto (problems whose output tiles
                        fill at most a quarter of the GPU -- half for the
                        32- and 64-column tiles of few-row and few-column
                        problems -- and have a long K use stream-K: every
                        cluster takes an equal contiguous share of the
                        (tile, K block) iterations), -1 = stream-K, 1 = one
                        pass per tile, n >= 2 = every tile split into n K
                        ranges (capped at the number of 128-byte K blocks and
                        at 2^29 / tiles units).  Problems with more than 2^29
                        output tiles return TCG_ERR_UNSUPPORTED.  Each unit that
                        computes part of a tile stores an fp32 partial in a
                        workspace owned by the library per (device, stream); a
                        second kernel sums each tile's partials in K order
                        (deterministic) into D.  Ignored with TCG_F16
                        accumulation. */
  int epilogue;      /* how 16-bit outputs (f16 / bf16 D, fp32 accumulation,
                        16-byte aligned D and ldd) leave TMEM: 0 = auto (1),
                        1 = tcgen05.ld .32x32b rows written to the staging tile
                        with st.shared.v4, 2 = tcgen05.ld .16x256b fragments
                        written with stmatrix .m8n8.x4 ("ldmatrix / stmatrix"
                        page).  Same values either way; other outputs ignore
                        it.  Anything else: TCG_ERR_INVALID. */
} tcg_gemm_args;

int tcg_gemm(const tcg_gemm_args* args, void* stream);

/* ---------------------------------------------------------------------------
 * Chained GEMM with the intermediate in tensor memory ("tcgen05.mma" page,
 * "Operands and repeat axes": the A operand may come from shared memory or
 * from TMEM).
 *
 *     C = A . B1            fp32 accumulation, rounded (RNE) to in_type
 *     E = C . B2            fp32 accumulation, stored as e_type
 *
 * A [M][K], B1 [N1][K] and B2 [N2][N1] are f16 or bf16 (in_type TCG_IN_F16 /
 * TCG_IN_BF16), all K-major with 16-byte aligned bases and leading
 * dimensions in elements (0 = packed) whose byte size is a multiple of 16;
 * E is row-major [M][lde] (0 = N2) with a 16-byte aligned base and row
 * stride (TCG_ERR_ALIGNMENT otherwise).  N1 is a multiple of 16 in [16, 256]
 * (TCG_ERR_INVALID otherwise).  The result equals two tcg_gemm calls with a
 * C of in_type in between, without C ever reaching global memory: each CTA
 * computes 128 rows of C into TMEM, rewrites them there as 16-bit pairs
 * (row m in lane m, element k in column k/2) and issues the second product's
 * MMAs with A read from TMEM, for 192-column tiles of E.  When there are
 * fewer 128-row tiles than SMs the E tiles are split into groups and each
 * group recomputes its rows of C.  With at least 16 row tiles and N1 >= 128
 * the CTAs of neighbouring row tiles run as clusters of two that load half of
 * every B1 / B2 tile each and share it by TMA multicast.  M == 0 or N2 == 0:
 * no-op; K == 0: E is zeroed.  One kernel launch; asynchronous on `stream`. */
int tcg_gemm_chain(tcg_input in_type, int64_t M, int64_t N1, int64_t N2, int64_t K,
                   const void* A, int64_t lda, const void* B1, int64_t ldb1,
                   const void* B2, int64_t ldb2, void* E, tcg_dtype e_type, int64_t lde,
                   void* stream);

/* ---------------------------------------------------------------------------
 * Block-scale layout (the scale-factor rearrangement step).
 *
 * The "tcgen05.mma" page places the scale of row r at TMEM lane r%32,
 * byte-column 4*(r//32)+sf, replicated in four 32-lane groups, which is what
 * one tcgen05.cp .32x128b.warpx4 produces from a 512-byte shared image in
 * which the scale of row r and K block kb sits at byte 16*(r%32) + 4*(r//32)
 * + kb.  The prepared image is, for every K step of 4 scale blocks (128 K
 * elements) and every tile of `tile_rows` rows, ceil(tile_rows/128) such
 * 512-byte chunks: [K step][tile][chunk][512 bytes].  Missing rows and K
 * blocks hold 127 (2^0).
 * ------------------------------------------------------------------------- */

/* Bytes of the image for `rows` rows, K elements, tiles of tile_rows rows. */
int64_t tcg_mxf8_scale_image_bytes(int64_t rows, int64_t K, int tile_rows);

/* The same for any block-scaled format (fmt TCG_IN_E4M3 .. TCG_IN_NVF4): a
 * ring stage covers 128 K (MX 8- and 6-bit formats) or 256 K (FP4), i.e. 4,
 * 8 (MXFP4) or 16 (NVFP4) scales per row, so the image is, per stage and
 * tile, ceil(tile_rows/128) x (1, 2 or 4) chunks of 512 bytes:
 * [stage][tile][group of 4 scales][chunk][512 B]; missing rows and scales
 * hold the scale of one (e8m0 127, E4M3 0x38).  -1 for a non-block-scaled
 * fmt or negative sizes. */
int64_t tcg_scale_image_bytes(tcg_input fmt, int64_t rows, int64_t K, int tile_rows);

/* tile_rows the GEMM uses for SFA (always 128 per CTA) and SFB (the N tile),
 * for a given block-scaled format, problem and cta_group request (0 = auto):
 * 256, or 384 for packed FP4 (TCG_IN_E2M1, TCG_IN_NVF4) on CTA pairs with
 * K-major B and at least 300 tiles of 256 x 384.  Depends on the arguments
 * alone (no device query).  TCG_ERR_INVALID for a format without block
 * scales. */
int tcg_tile_n(tcg_input fmt, int64_t M, int64_t N, int64_t K, tcg_major b_major, int cta_group);

/* tcg_tile_n for TCG_IN_E4M3. */
int tcg_mxf8_tile_n(int64_t M, int64_t N, int64_t K, tcg_major b_major, int cta_group);

/* Device-side rearrangement: `sf` plain [rows][ceil(K/32)] (device) -> `img`
 * (device, tcg_mxf8_scale_image_bytes bytes). */
int tcg_mxf8_prepare_scales(const uint8_t* sf, int64_t rows, int64_t K, int tile_rows,
                            uint8_t* img, void* stream);

/* Both images of one GEMM in a single launch: SFA [M][ceil(K/32)] -> SFA_img
 * with 128-row tiles, SFB [N][ceil(K/32)] -> SFB_img with tile_n-row tiles
 * (tcg_mxf8_tile_n).  The same result as two tcg_mxf8_prepare_scales calls;
 * M == 0 or N == 0 skips that matrix (its pointers may then be NULL). */
int tcg_mxf8_prepare_scales_ab(const uint8_t* SFA, int64_t M, uint8_t* SFA_img,
                               const uint8_t* SFB, int64_t N, int tile_n, uint8_t* SFB_img,
                               int64_t K, void* stream);

/* tcg_mxf8_prepare_scales_ab for any block-scaled format: plain scales of fmt
 * (e8m0 per 32, or unsigned E4M3 per 16 for TCG_IN_NVF4) into the images
 * tcg_gemm reads (sizes from tcg_scale_image_bytes; tile_n from
 * tcg_tile_n for the same format). */
int tcg_prepare_scales_ab(tcg_input fmt, const uint8_t* SFA, int64_t M, uint8_t* SFA_img,
                          const uint8_t* SFB, int64_t N, int tile_n, uint8_t* SFB_img,
                          int64_t K, void* stream);

/* ---------------------------------------------------------------------------
 * Status and configuration.
 * ------------------------------------------------------------------------- */

/* Synchronises `stream`, then returns and clears the current device's error
 * word: TCG_OK, TCG_ERR_TIMEOUT (a bounded wait ran out; the kernel returned
 * early, its output is incomplete) or TCG_ERR_CUDA. */
int tcg_check(void* stream);

/* Upper bound, in nanoseconds, of every mbarrier wait inside the kernels
 * launched after this call (default 2e9, i.e. 2 s; values < 1000 are
 * clamped).  Also settable through the TCG_WAIT_TIMEOUT_NS environment
 * variable at library load. */
void tcg_set_wait_timeout_ns(uint64_t ns);

const char* tcg_status_string(int status);

/* Text of the last CUDA error seen by this thread (empty if none). */
const char* tcg_last_error_string(void);

/* Number of kernels the most recent successful call on this thread queued. */
int tcg_last_launch_count(void);

/* How the most recent successful GEMM call on this thread was run (kernel
 * tile, CTA group, clusters, one pass / split-K / stream-K, operand swap), as
 * text for logs and tests; empty if the call queued nothing.  The string is
 * formatted by this call, owned by the library and valid until this thread's
 * next tcg_last_plan_string call. */
const char* tcg_last_plan_string(void);

/* Phase trace of the next GEMM kernel launched by this thread (tcg_gemm and
 * its wrappers; tcg_gemm_chain's kernel writes slots 0, 6, 7, 8 and 9 only).
 * Tracing is off otherwise and costs one untaken branch per stamp.  buf:
 * device memory of
 * max_ctas x 10 uint64 (8-byte aligned); CTA c (c < max_ctas) writes slots
 * [10c, 10c+10): globaltimer nanoseconds at 0 kernel entry, 1 barriers and
 * TMEM ready, 2 producer starts its first unit, 3 first unit's MMAs issued,
 * 4 last accumulator committed, 5 epilogue stores drained, 6 TMEM released;
 * slot 7 = units (tiles or tile parts) the CTA computed; slots 8 and 9 = the
 * SM's cycle counter (clock64) read right after the stamps of slots 0 and 6,
 * so (s9 - s8) / (s6 - s0) is the CTA's average SM clock in GHz.  Slots 3, 4
 * and 7 are written by the pair leader only (CTA pairs issue from the
 * leader).  No stamp sits inside the per-stage loops.
 * Untouched slots keep their contents.  buf = NULL with max_ctas = 0 cancels
 * a pending request. */
int tcg_trace_next(unsigned long long* buf, int max_ctas);

/* ---------------------------------------------------------------------------
 * Layout probes: single-CTA kernels that expose one tcgen05 / ldmatrix
 * mechanism each, so the tests can compare it bit for bit with the pages'
 * layout rules.  All buffers are device memory.
 * ------------------------------------------------------------------------- */

/* "tcgen05.ld / tcgen05.st" page example (Layout B) and the copy_async
 * round trip: 128 threads; thread t stores in[t*ncols .. +ncols) to TMEM lane
 * t with tcgen05.st .32x32b.x<ncols>, waits, reads it back with
 * tcgen05.ld .32x32b.x<ncols> into out.  ncols in {1,2,4,8,16,32,64,128}. */
int tcg_probe_tmem_roundtrip(const uint32_t* in, uint32_t* out, int ncols, void* stream);

/* "tcgen05.cp" page: fills a 1024-byte-aligned shared buffer with
 * `image_words` words of `image`, issues one tcgen05.cp of `shape`
 * (0 = 128x256b, 1 = 128x128b, 2 = 32x128b.warpx4, 3 = 4x256b; plus 4 for the
 * same shape with .b8x16.b4x16_p64 FP4 decompression, plus 8 for
 * .b8x16.b6x16_p32 FP6 decompression, "Native FP4/FP6 decompression": each
 * 16-byte source block of packed values and padding becomes sixteen
 * expanded bytes) with the descriptor (origin_bytes, ldo, sdo, swizzle 0..3),
 * waits on its commit and reads 128 lanes x 8 columns back with
 * tcgen05.ld .32x32b.x8 into out (128 x 8 words, lane-major; cells the copy
 * does not write hold 0xDEADBEEF).  image_words <= 12288; the walk must stay
 * inside the image, with every 8-row group it touches backed whole ("tcgen05.cp"
 * page: a 4-row region still needs the eight-row organisation's storage), else
 * TCG_ERR_INVALID before any launch. */
int tcg_probe_cp(const uint32_t* image, int image_words, int shape,
                 uint32_t origin_bytes, uint32_t ldo, uint32_t sdo, int swizzle,
                 uint32_t* out, void* stream);

/* "tcgen05.ld / tcgen05.st" page, native images: stores `in` (128 lanes x 32
 * columns, lane-major) with .32x32b.x32, then every warp loads lanes
 * [32w + half*16, +16) with tcgen05.ld.<shape>.x<num>; out receives, for
 * thread t, its registers at out[t*regs + r] (regs = registers per lane).
 * shape: 0 = 32x32b, 1 = 16x64b, 2 = 16x128b, 3 = 16x256b; num in {1,2,4} and
 * the larger repeats whose columns fit the image (32x32b up to 32, 16x64b up
 * to 16, 16x128b up to 8);
 * half in {0,1} (16-row shapes only). */
int tcg_probe_ld_shape(const uint32_t* in, int shape, int num, int half,
                       uint32_t* out, void* stream);

/* "tcgen05.mma" page example, generalised: one CTA; A (128 x K, K-major) and
 * B (N x K, K-major) f16/bf16 bytes are written into 128B-swizzled shared
 * memory with ordinary stores at the addresses the descriptor walk gives,
 * then K/16 tcgen05.mma kind::f16 (M=128, N, K=16) issues, one commit, and a
 * tcgen05.ld .32x32b drain into D (128 x N fp32).  K in {16..64} step 16,
 * N in {16..256} step 16.  is_bf16 selects the A/B format. */
int tcg_probe_mma_tile(const void* A, const void* B, int N, int K, int is_bf16,
                       float* D, void* stream);

/* "tcgen05.mma" page, "Weight-stationary and block scaling": the same tile as
 * tcg_probe_mma_tile issued with the weight-stationary opcode
 * tcgen05.mma.ws.cta_group::1.kind::f16 (M = 128, whose accumulator uses the
 * same lane-per-row Layout D as the dense form).  N in {64, 128, 256} (the
 * .ws shapes), K in {16, 32, 48, 64}. */
int tcg_probe_mma_tile_ws(const void* A, const void* B, int N, int K, int is_bf16, float* D, void* stream);

/* "tcgen05.mma" page, "Operands and repeat axes" (A "Shared or TMEM"; "A in
 * TMEM is packed according to its input format"; M = 128 uses Layout D): the
 * tile of tcg_probe_mma_tile with A read from tensor memory.  Thread t writes
 * row t of A (K f16 / bf16 values, two per 32-bit column, element 2c in the
 * low half of column c) to TMEM lane t with tcgen05.st .32x32b; K/16 MMAs
 * kind::f16 (M = 128, N) take A from columns [8j, 8j+8) of that image and B
 * (N x K, K-major) from a 128B-swizzled shared tile.  N in {16..256} step 16,
 * K in {16, 32, 48, 64}; D is 128 x N fp32, row-major. */
int tcg_probe_mma_tmem_a(const void* A, const void* B, int N, int K, int is_bf16, float* D, void* stream);

/* "tcgen05.mma" page, "Weight-stationary and block scaling": one
 * tcgen05.mma.ws.cta_group::1.kind::f16 tile of M = 64 (N in {64, 128, 256},
 * K in {16, 32, 48, 64}).  a_tmem = 0: A is 64 x K (row-major f16 / bf16),
 * written to a 128B-swizzled shared tile.  a_tmem = 1: A is the (2, 64, K)
 * two-bank image the page gives for M64 .ws with A in TMEM; thread t writes
 * bank t / 64, row t % 64 to TMEM lane t (two 16-bit values per column).  B is
 * N x K, K-major.  `out` receives the raw accumulator image: 128 lanes x N/2
 * fp32 columns, lane-major (out[lane * N/2 + column]). */
int tcg_probe_mma_ws64(const void* A, int a_tmem, const void* B, int N, int K, int is_bf16, uint32_t* out,
                       void* stream);

/* "tcgen05.mma" page, "Shared descriptors are byte-stride contracts" and
 * "swizzle=4": MMAs that read operands laid out by the caller.  One operand's
 * shared-memory image and the descriptors that walk it: */
typedef struct {
  const void* image;  /* device memory, 16-byte aligned: the operand's bytes exactly as
                         they must sit in shared memory from a 1024-byte aligned base */
  int bytes;          /* image size: a multiple of 16, at most 96 KiB */
  tcg_major major;    /* K-major or MN-major (the instruction descriptor's transpose bit) */
  uint32_t ldo, sdo;  /* descriptor leading / stride byte offsets (16-byte multiples < 2^18) */
  int swizzle;        /* the pages' logical mode 0..3; 4 (128-byte span, 32-byte atoms) is
                         required for, and only allowed with, TF32 MN-major */
  uint32_t start[8];  /* descriptor origin of MMA issue j, bytes from the image start
                         (16-byte multiples) */
} tcg_probe_operand;

/* One CTA zeroes two 96 KiB shared regions, copies a->image into the first
 * and b->image into the second, and one thread issues `ksteps` (1..8)
 * tcgen05.mma.cta_group::1 of kind::f16 (in_type TCG_IN_F16 / TCG_IN_BF16) or
 * kind::tf32 (TCG_IN_TF32), M = 128, N in {16..256} step 16, accumulation off
 * on the first issue only; issue j's descriptors are (region + start[j], ldo,
 * sdo, swizzle).  One commit, then D (128 x N fp32, row-major) is drained with
 * tcgen05.ld .32x32b.  Each issue multiplies 128 x 16 (16-bit) or 128 x 8
 * (TF32) of A by the same K of N rows of B.  The device computes no layout:
 * which element each step of the hardware walk reads is decided by the images
 * alone, so the result checks the caller's layout model.  Before any launch
 * the host rejects (TCG_ERR_INVALID) a walk that could leave its region under
 * either assignment of LDO and SDO. */
int tcg_probe_mma_image(const tcg_probe_operand* a, const tcg_probe_operand* b, tcg_input in_type, int N,
                        int ksteps, float* D, void* stream);

/* "ldmatrix / stmatrix" page example: x = 128 words viewed as (16,4,2) with
 * shared layout (16,4,2):(8,1,128); one warp issues two ldmatrix .m8n8.x2
 * into register slots {0,2} and {8,10} of a 12-word array preset to the
 * sentinel 4294966519; out is 32 x 12 words. */
int tcg_probe_ldmatrix_x2(const uint32_t* x, uint32_t* out, void* stream);

/* "ldmatrix / stmatrix" page, "Address providers and result owners" and
 * "Transpose and stores": one warp issues stmatrix .m8n8.x<count>[.trans].b16
 * (count 1, 2 or 4; trans 0 or 1) into a zeroed 1 KB shared buffer.  `regs`
 * (device, 128 words) gives lane l its registers regs[4l .. 4l+count);
 * `row_off` (device, 8*count words) gives the byte offset in the buffer of
 * row r of matrix m at row_off[8m + r]; lane l supplies row_off[l % (8*count)]
 * (so x1 / x2 repeat valid addresses).  Offsets must be multiples of 16 below
 * 1024: the kernel masks each with 1008, so no access leaves the buffer, and
 * a caller that breaks the rule simply gets a different image.  `out`
 * (device, 256 words) receives the buffer.  Returns TCG_ERR_INVALID for a
 * null pointer or another count. */
int tcg_probe_stmatrix(const uint32_t* regs, const uint32_t* row_off, int count, int trans, uint32_t* out,
                       void* stream);

/* "tcgen05.ld / tcgen05.st" page, "Split accesses: 16x32bx2": lane l owns
 * (access l/16, row l%16, column r); access 1 starts at the first address
 * plus the immediate (imm_lanes << 16) + imm_cols.  One CTA of 128 threads
 * allocates 64 columns; thread t stores in[32t .. 32t+32) (device, 128 x 32
 * words) to its TMEM lane t, columns 0..31, and zeroes columns 32..63.  Warp
 * w then issues, at lane 32w column 0,
 *     tcgen05.ld.16x32bx2.x<num>   -> out_ld[t*num + r]      (128 x num words)
 * and, at lane 32w column 32, stores the words 0x10000*t + r + 1 with
 *     tcgen05.st.16x32bx2.x<num>;
 * every thread then reads columns 32..63 of its lane into out_st[32t + c]
 * (128 x 32 words).  num in {1, 2, 4, 8}; (imm_lanes, imm_cols) one of
 * (16, 8), (16, 0), (0, 16), (16, 16) -- each keeps both accesses inside the
 * warp's 32 lanes and the allocation.  Anything else: TCG_ERR_INVALID, no
 * launch. */
int tcg_probe_ld_split(const uint32_t* in, int num, int imm_lanes, int imm_cols, uint32_t* out_ld,
                       uint32_t* out_st, void* stream);

/* Failure-detection probe: launches one CTA that waits on an mbarrier no one
 * arrives at, bounded by `timeout_ns`; the kernel records TCG_ERR_TIMEOUT in
 * the error word and returns.  Returns the launch status; tcg_check() then
 * reports the timeout. */
int tcg_probe_wait_timeout(uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TCG_H_ */
