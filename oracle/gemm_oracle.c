/*
 * Float64 CPU oracle for the tcgen05 swizzled GEMM path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (the plain definition of the contraction the tcgen05.mma
 * page describes, "tcgen05.mma" / "Operands and repeat axes", and its worked
 * example "four K16 issues for a 128x64x64 product", which checks against
 * a @ b.T):
 *
 *     D[m,n] = sum_k dec(A)[m,k] * dec(B)[k,n]
 *     S[m,n] = sum_k |dec(A)[m,k]| * |dec(B)[k,n]|
 *
 * For the block-scaled variant ("Weight-stationary and block scaling" on the
 * same page) every A element is multiplied by its row's scale for the K block
 * it falls in, and every B element by its column's:
 *
 *     dec(A)[m,k] = fp(A[m,k]) * scale(SFA[m, k/blk])
 *     dec(B)[k,n] = fp(B[k,n]) * scale(SFB[n, k/blk])
 *
 * with blk = 32 and e8m0 scales 2^(b-127) (the MX formats), or blk = 16 and
 * unsigned E4M3 scales (the NVFP4 format).
 *
 * where fp is the element format: E4M3 or E5M2 (one byte per element), E3M2 or
 * E2M3 (6 bits, packed four to three bytes) or E2M1 (4 bits, packed two to a
 * byte).
 *
 * S is the error scale the parity tolerance is stated against.
 *
 * Storage conventions (the page's "K-major rows enumerate M/N; MN-major rows
 * enumerate K"):  A K-major is M x K row-major, A MN-major is K x M
 * row-major; B K-major is N x K row-major, B MN-major is K x N row-major.
 * lda/ldb are the row strides of the stored matrices in elements.  Packed
 * formats store element i of the whole array (i = row * ld + column) in bits
 * [b*i, b*(i+1)) of the array read as one little-endian bit string (b = 4 or
 * 6): an FP4 byte holds element 2j in its low nibble and 2j+1 in its high one.
 *
 * The decoders below are written from the IEEE-754 binary16 / binary32, the
 * bfloat16 (truncated binary32), the OCP 8-bit floating point (E4M3FN, E5M2)
 * and the OCP microscaling (E3M2, E2M3, E2M1, E8M0) definitions by bit
 * manipulation; every value they produce is exact in float64.  FP32 storage is read exactly (no TF32 truncation): the GPU's TF32
 * rounding is covered by the tolerance, not by the oracle.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_E3M2 = 5, ORC_E2M3 = 6, ORC_E2M1 = 7 };
enum { ORC_K_MAJOR = 0, ORC_MN_MAJOR = 1 };

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_dec_f16(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^(1-15) */
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x400), e - 25); /* (1024+f) * 2^(e-15-10) */
  return s ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_dec_bf16(uint16_t h) {
  int s = h >> 15, e = (h >> 7) & 0xff, f = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)f, -133); /* f * 2^-7 * 2^(1-127) */
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x80), e - 134);
  return s ? -v : v;
}

/* binary32: 1 sign, 8 exponent (bias 127), 23 fraction bits. */
double oracle_dec_f32(uint32_t x) {
  int s = x >> 31, e = (x >> 23) & 0xff;
  uint32_t f = x & 0x7fffffu;
  double v;
  if (e == 0)
    v = ldexp((double)f, -149);
  else if (e == 255)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(f | 0x800000u), e - 150);
  return s ? -v : v;
}

/* E4M3FN: 1 sign, 4 exponent (bias 7), 3 fraction bits; S.1111.111 is NaN,
 * there is no infinity. */
double oracle_dec_e4m3(uint8_t x) {
  int s = x >> 7, e = (x >> 3) & 0xf, f = x & 7;
  double v;
  if (e == 15 && f == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)f, -9); /* f/8 * 2^(1-7) */
  else
    v = ldexp((double)(f | 8), e - 10); /* (8+f) * 2^(e-7-3) */
  return s ? -v : v;
}

/* E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE-like: exponent
 * 31 is infinity (fraction 0) or NaN. */
double oracle_dec_e5m2(uint8_t x) {
  int s = x >> 7, e = (x >> 2) & 0x1f, f = x & 3;
  double v;
  if (e == 31)
    v = f ? NAN : INFINITY;
  else if (e == 0)
    v = ldexp((double)f, -16); /* f/4 * 2^(1-15) */
  else
    v = ldexp((double)(f | 4), e - 17); /* (4+f) * 2^(e-15-2) */
  return s ? -v : v;
}

/* The OCP microscaling element formats have no infinity or NaN: every code is
 * a finite value (-1)^s * 2^(e-bias) * (1 + f/2^F), or 2^(1-bias) * f/2^F
 * when e == 0. */
static double dec_minifloat(unsigned x, int ebits, int fbits, int bias) {
  const int s = (x >> (ebits + fbits)) & 1;
  const int e = (x >> fbits) & ((1 << ebits) - 1);
  const int f = x & ((1 << fbits) - 1);
  const double v = e == 0 ? ldexp((double)f, 1 - bias - fbits) : ldexp((double)(f | (1 << fbits)), e - bias - fbits);
  return s ? -v : v;
}

/* E3M2 (FP6): 1 sign, 3 exponent (bias 3), 2 fraction bits. */
double oracle_dec_e3m2(uint8_t x) { return dec_minifloat(x & 0x3f, 3, 2, 3); }

/* E2M3 (FP6): 1 sign, 2 exponent (bias 1), 3 fraction bits. */
double oracle_dec_e2m3(uint8_t x) { return dec_minifloat(x & 0x3f, 2, 3, 1); }

/* E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 fraction bit. */
double oracle_dec_e2m1(uint8_t x) { return dec_minifloat(x & 0xf, 2, 1, 1); }

/* UE4M3: the E4M3FN encoding without its sign bit (scales are positive);
 * 0x7F is NaN, codes with the top bit set are not scales. */
double oracle_dec_ue4m3(uint8_t x) { return x & 0x80 ? NAN : oracle_dec_e4m3(x); }

/* E8M0: unsigned power of two 2^(b-127); 0xFF is NaN. */
double oracle_dec_e8m0(uint8_t b) {
  if (b == 0xff) return NAN;
  return ldexp(1.0, (int)b - 127);
}

/* Code of element idx of a packed array of `bits`-bit values (little-endian
 * bit string). */
static unsigned packed_code(const uint8_t* p, int64_t idx, int bits) {
  const int64_t bit = idx * bits;
  const int sh = (int)(bit & 7);
  unsigned two = (unsigned)p[bit >> 3];
  if (sh + bits > 8) two |= (unsigned)p[(bit >> 3) + 1] << 8; /* the value straddles two bytes */
  return (two >> sh) & ((1u << bits) - 1u);
}

static double dec_elem(const void* base, int type, int64_t idx) {
  switch (type) {
    case ORC_F32: return oracle_dec_f32(((const uint32_t*)base)[idx]);
    case ORC_F16: return oracle_dec_f16(((const uint16_t*)base)[idx]);
    case ORC_BF16: return oracle_dec_bf16(((const uint16_t*)base)[idx]);
    case ORC_E4M3: return oracle_dec_e4m3(((const uint8_t*)base)[idx]);
    case ORC_E5M2: return oracle_dec_e5m2(((const uint8_t*)base)[idx]);
    case ORC_E3M2: return oracle_dec_e3m2((uint8_t)packed_code((const uint8_t*)base, idx, 6));
    case ORC_E2M3: return oracle_dec_e2m3((uint8_t)packed_code((const uint8_t*)base, idx, 6));
    case ORC_E2M1: return oracle_dec_e2m1((uint8_t)packed_code((const uint8_t*)base, idx, 4));
  }
  return NAN;
}

enum { ORC_SF_E8M0 = 0, ORC_SF_UE4M3 = 1 };

typedef struct {
  int64_t M, N, K;
  int sf_block, sf_kind;
  const void* A; int a_type, a_major; int64_t lda;
  const void* B; int b_type, b_major; int64_t ldb;
  const uint8_t* SFA; int64_t ldsfa;
  const uint8_t* SFB; int64_t ldsfb;
  const int64_t* rows; int64_t nrows;
  double* Bd;          /* decoded B, K x N */
  double* D; double* S;
  int nthreads, tid;
} job_t;

static double dec_scale(uint8_t b, int kind) { return kind == ORC_SF_UE4M3 ? oracle_dec_ue4m3(b) : oracle_dec_e8m0(b); }

/* Step 1: decode (and scale) B into a dense K x N float64 matrix. */
static void* decode_b(void* p) {
  job_t* j = (job_t*)p;
  for (int64_t k = j->tid; k < j->K; k += j->nthreads) {
    for (int64_t n = 0; n < j->N; ++n) {
      int64_t idx = (j->b_major == ORC_K_MAJOR) ? n * j->ldb + k : k * j->ldb + n;
      double b = dec_elem(j->B, j->b_type, idx);
      if (j->SFB) b *= dec_scale(j->SFB[n * j->ldsfb + k / j->sf_block], j->sf_kind);
      j->Bd[k * j->N + n] = b;
    }
  }
  return NULL;
}

/* Step 2: for each requested output row m, the triple loop over k and n. */
static void* rows_job(void* p) {
  job_t* j = (job_t*)p;
  double* a = (double*)malloc(sizeof(double) * (size_t)(j->K > 0 ? j->K : 1));
  for (int64_t i = j->tid; i < j->nrows; i += j->nthreads) {
    int64_t m = j->rows ? j->rows[i] : i;
    for (int64_t k = 0; k < j->K; ++k) {
      int64_t idx = (j->a_major == ORC_K_MAJOR) ? m * j->lda + k : k * j->lda + m;
      double v = dec_elem(j->A, j->a_type, idx);
      if (j->SFA) v *= dec_scale(j->SFA[m * j->ldsfa + k / j->sf_block], j->sf_kind);
      a[k] = v;
    }
    double* d = j->D + i * j->N;
    double* s = j->S + i * j->N;
    for (int64_t n = 0; n < j->N; ++n) { d[n] = 0.0; s[n] = 0.0; }
    for (int64_t k = 0; k < j->K; ++k) {
      const double av = a[k];
      const double* brow = j->Bd + k * j->N;
      for (int64_t n = 0; n < j->N; ++n) {
        const double prod = av * brow[n];
        d[n] += prod;
        s[n] += fabs(prod);
      }
    }
  }
  free(a);
  return NULL;
}

static int run_threads(job_t* base, void* (*fn)(void*)) {
  int nt = base->nthreads;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nt);
  if (!th || !jobs) { free(th); free(jobs); return -2; }
  for (int t = 0; t < nt; ++t) {
    jobs[t] = *base;
    jobs[t].tid = t;
    if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) {
      /* fall back: run the remaining share on this thread */
      fn(&jobs[t]);
      th[t] = 0;
    }
  }
  for (int t = 0; t < nt; ++t)
    if (th[t]) pthread_join(th[t], NULL);
  free(th);
  free(jobs);
  return 0;
}

int oracle_num_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Computes the requested rows of D and S.
 *   rows == NULL: all M rows, written to D/S as M x N (row-major).
 *   rows != NULL: nrows rows; output row i is D row rows[i].
 * SFA/SFB may be NULL (no block scaling).  ldsfa/ldsfb are the row strides of
 * the plain [M][ceil(K/blk)] / [N][ceil(K/blk)] scale arrays; sf_block is blk
 * (32 or 16) and sf_kind the scale encoding (0 e8m0, 1 unsigned E4M3).  nthreads <= 0 uses all
 * online cores.  Returns 0, or a negative value on invalid arguments or
 * allocation failure.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void* A, int a_type, int a_major, int64_t lda,
                const void* B, int b_type, int b_major, int64_t ldb,
                const uint8_t* SFA, int64_t ldsfa,
                const uint8_t* SFB, int64_t ldsfb, int sf_block, int sf_kind,
                const int64_t* rows, int64_t nrows,
                double* D, double* S, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || !D || !S) return -1;
  if (sf_block != 16 && sf_block != 32) return -1;
  if (!rows) nrows = M;
  if (nrows == 0 || N == 0) return 0;
  if (K > 0 && (!A || !B)) return -1;
  if (nthreads <= 0) nthreads = oracle_num_threads();
  job_t base;
  memset(&base, 0, sizeof(base));
  base.M = M; base.N = N; base.K = K;
  base.A = A; base.a_type = a_type; base.a_major = a_major; base.lda = lda;
  base.B = B; base.b_type = b_type; base.b_major = b_major; base.ldb = ldb;
  base.SFA = SFA; base.ldsfa = ldsfa; base.SFB = SFB; base.ldsfb = ldsfb;
  base.sf_block = sf_block; base.sf_kind = sf_kind;
  base.rows = rows; base.nrows = nrows;
  base.D = D; base.S = S;
  base.nthreads = nthreads;
  base.Bd = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)N);
  if (!base.Bd) return -2;
  int rc = 0;
  if (K > 0) rc = run_threads(&base, decode_b);
  if (rc == 0) rc = run_threads(&base, rows_job);
  free(base.Bd);
  return rc;
}
