/*
 * mxoracle.c -- plain CPU oracle for the block-scaled (MX) matrix product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * path.
 *
 * What it computes (the plain definition, no blocking or fusion):
 *
 *   ref[i][j]   = sum_{k<K} fa(A[i][k]) * e8m0(As[i][k/32])
 *                         * fb(B[k][j]) * e8m0(Bs[j][k/32])
 *
 * fa, fb: element decoders; E4M3 for the headline path, E5M2, E2M3, E3M2
 * or E2M1 for the other formats of the same MX family.
 *   bound[i][j] = sum_{k<K} | same term |
 *
 * accumulated in IEEE double, k ascending.
 *
 * Sources:
 *   - "TLX API Quick Reference", section "Matrix Multiply (MMA)", row
 *     `tlx.async_dot_scaled`: the scaled product D = (A*scale_A) @ (B*scale_B)
 *     + D with FP8 operands.
 *   - "Tensor core operations", sections "2-CTA Scaled MMA" and "TMEM-backed
 *     MX Scales": operands in format "e4m3", one uint8 scale tensor per
 *     operand.
 *   - OCP Microscaling Formats (MX) specification v1.0, element format E4M3
 *     (bias 7, subnormals, max 448, S.1111.111 = NaN, no infinities) and
 *     scale format E8M0 (2^(s-127), s = 255 is NaN); one scale per block of
 *     32 consecutive elements along the reduction dimension.
 *
 * Layouts (all row-major, no padding):
 *   A  : M x K bytes        As : M x (K/32) bytes
 *   B  : K x N bytes        Bs : N x (K/32) bytes
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread -ffp-contract=off
 * (-ffp-contract=off keeps every multiply and add separately rounded on
 * every host, so the result does not depend on whether the compiler fuses.)
 *
 * Parity of the GPU path against this oracle is governed by a tolerance; the
 * order in which the GPU accumulates is not modelled here.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* Element and scale decoders, written from the format definitions.       */
/* ---------------------------------------------------------------------- */

/* E4M3: bit 7 sign, bits 6..3 exponent E (bias 7), bits 2..0 mantissa m.
 *   E == 0          : (-1)^s * m * 2^-9            (subnormal, m/8 * 2^-6)
 *   E != 0          : (-1)^s * (1 + m/8) * 2^(E-7)
 *   E == 15, m == 7 : NaN (no infinities in this format)                  */
double mxo_e4m3(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(8.0 + (double)m, e - 7 - 3);
  return s ? -v : v;
}

/* The other element formats of the same MX family (OCP MX v1.0), one code
 * per byte; the sub-byte formats use the low bits of the byte and ignore
 * the rest.
 *
 * E5M2: bit 7 sign, bits 6..2 exponent E (bias 15), bits 1..0 mantissa m.
 *   E == 0  : (-1)^s * m/4 * 2^-14          (subnormal)
 *   E == 31 : +-inf when m == 0, else NaN
 *   else    : (-1)^s * (1 + m/4) * 2^(E-15)                               */
double mxo_e5m2(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 2) & 31;
  int m = code & 3;
  double v;
  if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
  if (e == 0)
    v = ldexp((double)m, -16);
  else
    v = ldexp(4.0 + (double)m, e - 15 - 2);
  return s ? -v : v;
}

/* Sub-byte formats with sign bit at position (ebits + mbits), exponent
 * bias b, no infinities or NaN:
 *   E == 0 : (-1)^s * m / 2^mbits * 2^(1-b)        (subnormal)
 *   else   : (-1)^s * (1 + m / 2^mbits) * 2^(E-b)
 * E2M3 (FP6): ebits 2, mbits 3, bias 1 (max 7.5)
 * E3M2 (FP6): ebits 3, mbits 2, bias 3 (max 28)
 * E2M1 (FP4): ebits 2, mbits 1, bias 1 (max 6)                           */
static double mxo_small(uint8_t code, int ebits, int mbits, int bias) {
  int s = (code >> (ebits + mbits)) & 1;
  int e = (code >> mbits) & ((1 << ebits) - 1);
  int m = code & ((1 << mbits) - 1);
  double v;
  if (e == 0)
    v = ldexp((double)m, 1 - bias - mbits);
  else
    v = ldexp((double)((1 << mbits) + m), e - bias - mbits);
  return s ? -v : v;
}
double mxo_e2m3(uint8_t code) { return mxo_small(code, 2, 3, 1); }
double mxo_e3m2(uint8_t code) { return mxo_small(code, 3, 2, 3); }
double mxo_e2m1(uint8_t code) { return mxo_small(code, 2, 1, 1); }

/* element format ids: 0 E4M3, 1 E5M2, 2 E2M3, 3 E3M2, 4 E2M1 */
double mxo_decode(int fmt, uint8_t code) {
  switch (fmt) {
    case 0: return mxo_e4m3(code);
    case 1: return mxo_e5m2(code);
    case 2: return mxo_e2m3(code);
    case 3: return mxo_e3m2(code);
    case 4: return mxo_e2m1(code);
    default: return NAN;
  }
}

/* E8M0: an unsigned biased exponent with no sign and no mantissa.
 *   s in [0, 254] : 2^(s - 127)     s == 255 : NaN                        */
double mxo_e8m0(uint8_t code) {
  if (code == 255) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* ---------------------------------------------------------------------- */
/* The product, for a set of full output rows.                             */
/* ---------------------------------------------------------------------- */

typedef struct {
  int64_t M, N, K;
  const uint8_t *A, *As, *B, *Bs;
  const int64_t *rows; /* which rows of C to produce */
  int64_t nrows;
  double *ref, *bound; /* nrows x N each */
  const double *lut_a, *lut_b, *lut_e8m0;
  int64_t r_begin, r_end; /* this worker's share of `rows` */
} rows_job;

static void *rows_worker(void *arg) {
  rows_job *jb = (rows_job *)arg;
  const int64_t N = jb->N, K = jb->K, KB = K / 32;
  for (int64_t r = jb->r_begin; r < jb->r_end; ++r) {
    const int64_t i = jb->rows[r];
    double *acc = jb->ref + r * N;
    double *bnd = jb->bound + r * N;
    for (int64_t j = 0; j < N; ++j) {
      acc[j] = 0.0;
      bnd[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
      /* a = fa(A[i][k]) * e8m0(As[i][k/32]) */
      const double a = jb->lut_a[jb->A[i * K + k]] *
                       jb->lut_e8m0[jb->As[i * KB + k / 32]];
      const uint8_t *brow = jb->B + k * N;
      for (int64_t j = 0; j < N; ++j) {
        /* b = fb(B[k][j]) * e8m0(Bs[j][k/32]) */
        const double b =
            jb->lut_b[brow[j]] * jb->lut_e8m0[jb->Bs[j * KB + k / 32]];
        const double t = a * b;
        acc[j] += t;
        bnd[j] += fabs(t);
      }
    }
  }
  return NULL;
}

static void build_luts(int fa, int fb, double *la, double *lb, double *l8) {
  for (int c = 0; c < 256; ++c) {
    la[c] = mxo_decode(fa, (uint8_t)c);
    lb[c] = mxo_decode(fb, (uint8_t)c);
    l8[c] = mxo_e8m0((uint8_t)c);
  }
}

static int bad_fmt(int f) { return f < 0 || f > 4; }

/* Full rows `rows[0..nrows)` of the product, A's elements in format fa and
 * B's in fb.  ref and bound are nrows x N.  Returns 0 on success, -1 on a
 * bad argument. */
int mxo_rows_fmt(int64_t M, int64_t N, int64_t K, const uint8_t *A,
                 const uint8_t *As, const uint8_t *B, const uint8_t *Bs,
                 int64_t nrows, const int64_t *rows, double *ref, double *bound,
                 int nthreads, int fa, int fb) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || nrows < 0) return -1;
  if (bad_fmt(fa) || bad_fmt(fb)) return -1;
  for (int64_t r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return -1;
  double la[256], lb[256], l8[256];
  build_luts(fa, fb, la, lb, l8);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
  rows_job *jobs = (rows_job *)calloc((size_t)nthreads, sizeof(rows_job));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tid) {
    free(jobs);
    free(tid);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    rows_job *jb = &jobs[t];
    jb->M = M; jb->N = N; jb->K = K;
    jb->A = A; jb->As = As; jb->B = B; jb->Bs = Bs;
    jb->rows = rows; jb->nrows = nrows;
    jb->ref = ref; jb->bound = bound;
    jb->lut_a = la; jb->lut_b = lb; jb->lut_e8m0 = l8;
    jb->r_begin = nrows * t / nthreads;
    jb->r_end = nrows * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, rows_worker, &jobs[t]) != 0) break;
    started = t;
  }
  rows_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  /* any share whose thread could not start runs here */
  for (int t = started + 1; t < nthreads; ++t) rows_worker(&jobs[t]);
  free(jobs);
  free(tid);
  return 0;
}

/* ---------------------------------------------------------------------- */
/* The product at individual points (i, j): for checking sampled outputs.  */
/* ---------------------------------------------------------------------- */

typedef struct {
  int64_t N, K;
  const uint8_t *A, *As, *B, *Bs;
  const int64_t *I, *J;
  double *ref, *bound;
  const double *lut_a, *lut_b, *lut_e8m0;
  int64_t p_begin, p_end;
} points_job;

static void *points_worker(void *arg) {
  points_job *jb = (points_job *)arg;
  const int64_t N = jb->N, K = jb->K, KB = K / 32;
  for (int64_t p = jb->p_begin; p < jb->p_end; ++p) {
    const int64_t i = jb->I[p], j = jb->J[p];
    double acc = 0.0, bnd = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = jb->lut_a[jb->A[i * K + k]] *
                       jb->lut_e8m0[jb->As[i * KB + k / 32]];
      const double b = jb->lut_b[jb->B[k * N + j]] *
                       jb->lut_e8m0[jb->Bs[j * KB + k / 32]];
      const double t = a * b;
      acc += t;
      bnd += fabs(t);
    }
    jb->ref[p] = acc;
    jb->bound[p] = bnd;
  }
  return NULL;
}

int mxo_points_fmt(int64_t M, int64_t N, int64_t K, const uint8_t *A,
                   const uint8_t *As, const uint8_t *B, const uint8_t *Bs,
                   int64_t npts, const int64_t *I, const int64_t *J, double *ref,
                   double *bound, int nthreads, int fa, int fb) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || npts < 0) return -1;
  if (bad_fmt(fa) || bad_fmt(fb)) return -1;
  for (int64_t p = 0; p < npts; ++p)
    if (I[p] < 0 || I[p] >= M || J[p] < 0 || J[p] >= N) return -1;
  double la[256], lb[256], l8[256];
  build_luts(fa, fb, la, lb, l8);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > npts) nthreads = npts > 0 ? (int)npts : 1;
  points_job *jobs = (points_job *)calloc((size_t)nthreads, sizeof(points_job));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !tid) {
    free(jobs);
    free(tid);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    points_job *jb = &jobs[t];
    jb->N = N; jb->K = K;
    jb->A = A; jb->As = As; jb->B = B; jb->Bs = Bs;
    jb->I = I; jb->J = J;
    jb->ref = ref; jb->bound = bound;
    jb->lut_a = la; jb->lut_b = lb; jb->lut_e8m0 = l8;
    jb->p_begin = npts * t / nthreads;
    jb->p_end = npts * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, points_worker, &jobs[t]) != 0) break;
    started = t;
  }
  points_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) points_worker(&jobs[t]);
  free(jobs);
  free(tid);
  return 0;
}

/* E4M3 x E4M3, the format of the headline path */
int mxo_rows(int64_t M, int64_t N, int64_t K, const uint8_t *A,
             const uint8_t *As, const uint8_t *B, const uint8_t *Bs,
             int64_t nrows, const int64_t *rows, double *ref, double *bound,
             int nthreads) {
  return mxo_rows_fmt(M, N, K, A, As, B, Bs, nrows, rows, ref, bound, nthreads, 0, 0);
}

int mxo_points(int64_t M, int64_t N, int64_t K, const uint8_t *A,
               const uint8_t *As, const uint8_t *B, const uint8_t *Bs,
               int64_t npts, const int64_t *I, const int64_t *J, double *ref,
               double *bound, int nthreads) {
  return mxo_points_fmt(M, N, K, A, As, B, Bs, npts, I, J, ref, bound, nthreads, 0, 0);
}

/* ---------------------------------------------------------------------- */
/* Output rounding: double -> binary32 / bfloat16, round to nearest even.  */
/* ---------------------------------------------------------------------- */

/* binary32: the C conversion rounds to nearest-even under the default
 * floating-point environment (overflow gives +-inf). */
float mxo_round_f32(double x) { return (float)x; }

/* bfloat16 (1 sign, 8 exponent bits, 7 stored mantissa bits), written out
 * from its definition: keep 8 significant bits, round to nearest, ties to
 * even, values past the largest finite bfloat16 become infinities, results
 * below 2^-126 keep 8 - (extra exponent) bits (gradual underflow).
 * Returns the 16-bit pattern. */
uint16_t mxo_round_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double ax = fabs(x);
  if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
  if (isinf(x)) return (uint16_t)(sign | 0x7F80u);
  if (ax == 0.0) return sign;
  int e;
  (void)frexp(ax, &e); /* ax = f * 2^e, f in [0.5, 1) -> unbiased exp e-1 */
  int ue = e - 1;
  if (ue < -126) ue = -126; /* subnormal range: fixed quantum 2^-133 */
  /* quantum of the 8-bit significand at this exponent */
  double q = ldexp(1.0, ue - 7);
  double n = nearbyint(ax / q); /* ax/q is exact: a power-of-2 scaling */
  double r = n * q;             /* rounded magnitude (may carry to 2^(ue+1)) */
  if (r == 0.0) return sign;    /* underflow to a signed zero */
  /* largest finite bfloat16: (2 - 2^-7) * 2^127 */
  if (r > ldexp(255.0, 127 - 7)) return (uint16_t)(sign | 0x7F80u);
  /* encode r */
  int re;
  (void)frexp(r, &re);
  int rexp = re - 1;
  uint16_t bits;
  if (rexp < -126) {
    /* subnormal: r = mant * 2^-133 with mant < 128 */
    bits = (uint16_t)(int)ldexp(r, 133);
  } else {
    double frac = ldexp(r, -rexp) - 1.0; /* in [0,1) */
    bits = (uint16_t)(((rexp + 127) << 7) | (int)ldexp(frac, 7));
  }
  return (uint16_t)(sign | bits);
}

void mxo_round_bf16_array(const double *x, uint16_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = mxo_round_bf16(x[i]);
}

/* ---------------------------------------------------------------------- */
/* MX quantization of a real matrix to E4M3 codes with E8M0 block scales.  */
/* ---------------------------------------------------------------------- */
/*
 * Per block of 32 consecutive values x_0..x_31 (along a row, or down a
 * column), the block-scaling recipe of the inputs' generator, which is the
 * OCP Microscaling Formats v1.0 conversion with an E4M3 maximum of 448:
 *   amax  = max |x_i|
 *   scale = clamp(127 + ceil(log2(amax / 448)), 0, 254), and 127 if amax = 0
 *   code_i = E4M3 code nearest to clamp(x_i * 2^(127 - scale), -448, 448),
 *            ties to even (the sign of x_i kept, also for zero)
 * Written from those definitions in double: every step is exact except the
 * final round-to-nearest-even, which rint() performs on an exact value.
 * Inputs must be finite.
 */

/* smallest integer t with amax <= 448 * 2^t, for amax > 0 (exact) */
static int ceil_log2_over_448(double amax) {
  int E;
  const double f = frexp(amax, &E); /* amax = f * 2^E, f in [0.5, 1) */
  /* 448 * 2^t = 0.875 * 2^(t + 9) */
  return f <= 0.875 ? E - 9 : E - 8;
}

uint8_t mxo_e4m3_rne(double y) {
  const uint8_t sign = signbit(y) ? 0x80u : 0u;
  double a = fabs(y);
  if (a > 448.0) a = 448.0;
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9 (q = 8 is the smallest normal) */
    const double q = rint(ldexp(a, 9));
    return (uint8_t)(sign | (uint8_t)q);
  }
  int E;
  (void)frexp(a, &E);          /* a in [2^(E-1), 2^E) */
  int e = E - 1;               /* unbiased exponent */
  double q = rint(ldexp(a, 3 - e)) - 8.0; /* mantissa in eighths */
  if (q >= 8.0) {
    q = 0.0;
    e += 1;
  }
  return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)q);
}

/*
 * Stochastic rounding to E4M3 ("TLX API Quick Reference", section "Utility",
 * row `tlx.stoch_round`: FP32 -> FP8 with random bits the caller supplies).
 * The pages do not say how the random bits are used; the reading taken here
 * is the textbook one.  |y| (clamped to 448) lies between two adjacent E4M3
 * magnitudes lo <= |y| < lo + q, q the E4M3 spacing at |y| (2^(e-3) in the
 * binade [2^e, 2^(e+1)), 2^-9 below 2^-6).  With one random 32-bit word r per
 * value the result is lo + q when r < 2^32 * (|y| - lo) / q and lo otherwise:
 * it rounds away from zero with probability (|y| - lo) / q, to within 2^-32.
 * The sign is kept, also for zero.  Every step below is exact in double.
 */
uint8_t mxo_e4m3_sr(double y, uint32_t r) {
  const uint8_t sign = signbit(y) ? 0x80u : 0u;
  double a = fabs(y);
  if (a > 448.0) a = 448.0;
  if (a == 0.0) return sign;
  int E;
  (void)frexp(a, &E);        /* a in [2^(E-1), 2^E) */
  int e = E - 1;
  if (e < -6) e = -6;        /* below 2^-6 the grid is the subnormal one */
  const double q = ldexp(1.0, e - 3);
  const double lo = floor(a / q) * q;
  const double frac = (a - lo) / q; /* in [0, 1) */
  const double mag = (double)r < ldexp(frac, 32) ? lo + q : lo;
  return (uint8_t)(sign | mxo_e4m3_rne(mag)); /* mag is on the grid: its own code */
}

/* x: R x C row-major values.  along_cols = 0: blocks of 32 along each row
 * (C % 32 == 0), scales R x (C/32); along_cols = 1: blocks of 32 down each
 * column (R % 32 == 0), scales C x (R/32), row j holding column j's scales.
 * codes: R x C.  rbits: NULL for round-to-nearest-even, else R x C random
 * words (row-major, the same index as x) for stochastic rounding of the
 * scaled value taken as an FP32 number.  Returns 0, or -1 on a bad
 * argument. */
static int quantize_e4m3(int64_t R, int64_t C, const double *x, int along_cols,
                         const uint32_t *rbits, uint8_t *codes, uint8_t *scales) {
  if (R < 0 || C < 0 || (along_cols ? R % 32 : C % 32) != 0) return -1;
  const int64_t nblk = along_cols ? C * (R / 32) : R * (C / 32);
  for (int64_t b = 0; b < nblk; ++b) {
    /* element i of block b at x[base + i * step] */
    int64_t base, step;
    if (along_cols) {
      const int64_t j = b / (R / 32), rb = b % (R / 32);
      base = rb * 32 * C + j;
      step = C;
    } else {
      const int64_t r = b / (C / 32), cb = b % (C / 32);
      base = r * C + cb * 32;
      step = 1;
    }
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      const double a = fabs(x[base + i * step]);
      if (a > amax) amax = a;
    }
    int s = 127;
    if (amax > 0.0) {
      s = 127 + ceil_log2_over_448(amax);
      if (s < 0) s = 0;
      if (s > 254) s = 254;
    }
    scales[b] = (uint8_t)s; /* b enumerates blocks in the scales' own order */
    for (int i = 0; i < 32; ++i) {
      const int64_t at = base + i * step;
      const double y = ldexp(x[at], 127 - s);
      codes[at] = rbits ? mxo_e4m3_sr((double)(float)y, rbits[at]) : mxo_e4m3_rne(y);
    }
  }
  return 0;
}

int mxo_quantize_e4m3(int64_t R, int64_t C, const double *x, int along_cols, uint8_t *codes,
                      uint8_t *scales) {
  return quantize_e4m3(R, C, x, along_cols, NULL, codes, scales);
}

int mxo_quantize_e4m3_sr(int64_t R, int64_t C, const double *x, int along_cols,
                         const uint32_t *rbits, uint8_t *codes, uint8_t *scales) {
  if (!rbits) return -1;
  return quantize_e4m3(R, C, x, along_cols, rbits, codes, scales);
}
