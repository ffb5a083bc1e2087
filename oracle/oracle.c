/*
 * oracle.c -- plain, slow, CPU reference for FP8 quantization and scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference legs load this library. The CUDA library never
 * includes, links or calls it, and it includes nothing from the CUDA library.
 *
 * Every function follows a definition from the source pages:
 *   [Family]   "07 -- The FP8 Family: E4M3, E5M2, and Per-Block Scaling"
 *   [Serving]  "FP8 Mixed-Precision Serving in Production: Comparing E4M3 vs. E5M2 ..."
 *   [Guide]    "FP8 Serving" learning guide
 *   [LowPrec]  "Low precision: FP8, FP4, and microscaling"
 * Where the pages leave a step open, the reading taken is stated at the function.
 *
 * Arithmetic conventions: all scale arithmetic is single-precision IEEE with
 * round-to-nearest-even (the build uses -ffp-contract=off and no fast-math);
 * exact values (decoded codes, reference sums) are carried in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_E4M3 0
#define ORC_E5M2 1

#define ORC_GRAN_TENSOR 0
#define ORC_GRAN_TOKEN 1
#define ORC_GRAN_TILE_1x128 2
#define ORC_GRAN_BLOCK_128x128 3
#define ORC_GRAN_MX32 4
#define ORC_GRAN_CHANNEL 5

#define ORC_SF_LINEAR 0
#define ORC_SF_TILED 1

/* ------------------------------------------------------------------ */
/* parallel-for over [0, n) with plain pthreads                         */
/* ------------------------------------------------------------------ */
typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi, int tid);

typedef struct {
  range_fn fn;
  void *ctx;
  int64_t lo, hi;
  int tid;
} job_t;

static void *job_main(void *p) {
  job_t *j = (job_t *)p;
  if (j->lo < j->hi) j->fn(j->ctx, j->lo, j->hi, j->tid);
  return NULL;
}

int orc_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

static int resolve_threads(int nthreads) {
  if (nthreads <= 0) nthreads = orc_default_threads();
  if (nthreads > 256) nthreads = 256;
  return nthreads;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx) {
  nthreads = resolve_threads(nthreads);
  if (n <= 0) return;
  if ((int64_t)nthreads > n) nthreads = (int)n;
  pthread_t th[256];
  job_t jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].fn = fn;
    jobs[t].ctx = ctx;
    jobs[t].lo = (int64_t)t * per;
    jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
    jobs[t].tid = t;
  }
  for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, job_main, &jobs[t]);
  job_main(&jobs[0]);
  for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* bf16 <-> fp32                                                        */
/* ------------------------------------------------------------------ */
static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round an fp32 value to bf16, nearest with ties to even on the 16 dropped bits. */
static uint16_t f32_to_bf16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t keep = u >> 16;
  uint32_t drop = u & 0xffffu;
  if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

float orc_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }
uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16_rn(f); }

/* ------------------------------------------------------------------ */
/* decode: [Family] "The two shapes" bit layout; [Serving] "The Mathematics  */
/* of FP8" (bias 15 and IEEE inf/NaN for E5M2).                         */
/* ------------------------------------------------------------------ */
double orc_decode(uint32_t code, int fmt) {
  code &= 0xffu;
  double sign = (code & 0x80u) ? -1.0 : 1.0;
  if (fmt == ORC_E4M3) {
    int E = (int)((code >> 3) & 0xfu), M = (int)(code & 7u);
    if (E == 15 && M == 7) return NAN; /* S1111111: the only NaN, no infinities */
    if (E == 0) return sign * ldexp((double)M / 8.0, -6);
    return sign * ldexp(1.0 + (double)M / 8.0, E - 7);
  }
  /* E5M2. Subnormals follow the IEEE analogue 2^-14 * M/4 (the pages print only
     the normal formula). */
  int E = (int)((code >> 2) & 0x1fu), M = (int)(code & 3u);
  if (E == 31) return M ? NAN : sign * INFINITY;
  if (E == 0) return sign * ldexp((double)M / 4.0, -14);
  return sign * ldexp(1.0 + (double)M / 4.0, E - 15);
}

int orc_is_nan_code(uint32_t code, int fmt) {
  code &= 0x7fu;
  if (fmt == ORC_E4M3) return code == 0x7fu;
  return code > 0x7cu;
}

static uint32_t max_code(int fmt) { return fmt == ORC_E4M3 ? 0x7eu : 0x7bu; }
static uint8_t nan_code(int fmt) { return fmt == ORC_E4M3 ? 0x7f : 0x7f; }

double orc_fmt_max(int fmt) { return orc_decode(max_code(fmt), fmt); }

/* ------------------------------------------------------------------ */
/* encode (i): nearest finite value of the format, found by search over the  */
/* sorted table of non-negative finite values; ties go to the code whose     */
/* mantissa LSB is 0; beyond the largest finite value the result saturates   */
/* to it ("satfinite", [LowPrec] qdq_e4m3 listing: clamp instead of inf).    */
/* The sign of zero is kept.                                                 */
/* ------------------------------------------------------------------ */
static double g_tab[2][128];
static pthread_once_t g_tab_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
  for (int f = 0; f < 2; ++f)
    for (uint32_t c = 0; c <= max_code(f); ++c) g_tab[f][c] = orc_decode(c, f);
}

uint8_t orc_encode_nearest(float xf, int fmt) {
  pthread_once(&g_tab_once, build_tables);
  double x = (double)xf;
  if (isnan(x)) return nan_code(fmt);
  uint8_t sgn = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  const double *t = g_tab[fmt];
  int hi = (int)max_code(fmt);
  if (a >= t[hi]) return (uint8_t)(sgn | hi);
  int lo = 0; /* invariant: t[lo] <= a < t[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (t[mid] <= a)
      lo = mid;
    else
      hi = mid;
  }
  double dl = a - t[lo], dh = t[hi] - a; /* both exact in double */
  int c;
  if (dl < dh)
    c = lo;
  else if (dh < dl)
    c = hi;
  else
    c = (lo & 1) ? hi : lo;
  return (uint8_t)(sgn | c);
}

/* ------------------------------------------------------------------ */
/* encode (ii): the binade method of [Guide] ("find the binade, round the    */
/* mantissa to 3 or 2 bits"), done on the integer significand with ties to   */
/* even; below the smallest normal the quantum is fixed (2^-9 for E4M3,      */
/* 2^-16 for E5M2); the result then saturates to the largest finite code.    */
/* ------------------------------------------------------------------ */
uint8_t orc_encode_binade(float xf, int fmt) {
  uint32_t u;
  memcpy(&u, &xf, 4);
  uint8_t sgn = (u >> 31) ? 0x80 : 0;
  uint32_t ex = (u >> 23) & 0xffu, fr = u & 0x7fffffu;
  int mb = fmt == ORC_E4M3 ? 3 : 2;
  int bias = fmt == ORC_E4M3 ? 7 : 15;
  uint64_t maxc = max_code(fmt);
  if (ex == 0xffu) return fr ? nan_code(fmt) : (uint8_t)(sgn | maxc);
  if (ex == 0 && fr == 0) return sgn;
  uint64_t sig;
  int e2; /* |x| = sig * 2^e2 */
  if (ex == 0) {
    sig = fr;
    e2 = -149;
  } else {
    sig = fr | 0x800000u;
    e2 = (int)ex - 150;
  }
  int msb = 63 - __builtin_clzll(sig);
  int E = e2 + msb; /* binade: 2^E <= |x| < 2^(E+1) */
  int emin = 1 - bias;
  int qexp = (E < emin ? emin : E) - mb; /* spacing of the format in this binade */
  int shift = qexp - e2;                 /* > 0 for every finite fp32 input */
  uint64_t n;
  if (shift >= 64) {
    n = 0;
  } else {
    n = sig >> shift;
    uint64_t rem = sig & ((1ull << shift) - 1ull);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (n & 1ull))) n += 1;
  }
  uint64_t code;
  if (E < emin)
    code = n; /* subnormal codes are the integer count of quanta */
  else
    code = ((uint64_t)(E + bias) << mb) + (n - (1ull << mb)); /* carry moves into the exponent */
  if (code > maxc) code = maxc;
  return (uint8_t)(sgn | (uint8_t)code);
}

/* Agreement of the two encoders over fp32 bit patterns [start, start+count). */
typedef struct {
  uint64_t start;
  int fmt;
  const uint8_t *codes; /* NULL: compare encoders; else compare against these */
  int64_t bad[256];
  uint64_t first[256];
} cmp_ctx;

static int codes_equal(uint8_t a, uint8_t b, int fmt) {
  if (orc_is_nan_code(a, fmt) && orc_is_nan_code(b, fmt)) return 1;
  return a == b;
}

static void cmp_range(void *p, int64_t lo, int64_t hi, int tid) {
  cmp_ctx *c = (cmp_ctx *)p;
  int64_t bad = 0;
  uint64_t first = UINT64_MAX;
  for (int64_t i = lo; i < hi; ++i) {
    uint32_t bits = (uint32_t)(c->start + (uint64_t)i);
    float x;
    memcpy(&x, &bits, 4);
    uint8_t e1 = orc_encode_nearest(x, c->fmt);
    uint8_t e2 = c->codes ? c->codes[i] : orc_encode_binade(x, c->fmt);
    if (!codes_equal(e1, e2, c->fmt)) {
      if (first == UINT64_MAX) first = c->start + (uint64_t)i;
      ++bad;
    }
  }
  c->bad[tid] = bad;
  c->first[tid] = first;
}

static int64_t run_cmp(uint64_t start, uint64_t count, int fmt, const uint8_t *codes, int nthreads,
                       uint64_t *first_bad) {
  cmp_ctx c;
  memset(&c, 0, sizeof c);
  for (int i = 0; i < 256; ++i) c.first[i] = UINT64_MAX;
  c.start = start;
  c.fmt = fmt;
  c.codes = codes;
  parallel_for((int64_t)count, nthreads, cmp_range, &c);
  int64_t bad = 0;
  uint64_t first = UINT64_MAX;
  for (int i = 0; i < 256; ++i) {
    bad += c.bad[i];
    if (c.first[i] < first) first = c.first[i];
  }
  if (first_bad) *first_bad = first;
  return bad;
}

int64_t orc_encoders_disagree(uint64_t start, uint64_t count, int fmt, int nthreads, uint64_t *first_bad) {
  return run_cmp(start, count, fmt, NULL, nthreads, first_bad);
}

/* codes[i] is checked against the encoding of the fp32 pattern start+i. */
int64_t orc_check_codes(uint64_t start, uint64_t count, int fmt, const uint8_t *codes, int nthreads,
                        uint64_t *first_bad) {
  return run_cmp(start, count, fmt, codes, nthreads, first_bad);
}

void orc_encode_array(const float *x, int64_t n, int fmt, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_encode_nearest(x[i], fmt);
}

void orc_decode_array(const uint8_t *c, int64_t n, int fmt, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_decode(c[i], fmt);
}

/* ------------------------------------------------------------------ */
/* scales                                                               */
/* ------------------------------------------------------------------ */
/* V_max of the target format: 448 for E4M3 ([Serving] per-tensor static   */
/* scaling), 57344 for E5M2 (its largest finite value).                   */
static float vmax_f(int fmt) { return fmt == ORC_E4M3 ? 448.0f : 57344.0f; }

/* s = amax / V_max in fp32 (round to nearest); s_inv = 1/s in fp32. A zero
   or non-finite s_inv (all-zero group, or a group so small that 1/s
   overflows) is replaced by 0, so that every code of the group is +-0. */
static void scale_from_amax(float amax, int fmt, float *s, float *s_inv) {
  float sv = amax / vmax_f(fmt);
  float si = 1.0f / sv;
  if (sv == 0.0f || !isfinite(si)) si = 0.0f;
  *s = sv;
  *s_inv = si;
}

/* MX: one UE8M0 scale per 32 consecutive elements ([LowPrec] microscaling;
   [Family] granularity ladder). The pages fix neither the rounding of the
   shared exponent nor how amax maps to it; the reading taken is
   e = ceil(log2(fp32(amax / V_max))), clamped to [-127, 127] (-127 for an
   all-zero block), so that the largest element lands in (V_max/2, V_max].
   ceil(log2 t) is read from the bits of t. */
static int mx_exponent(float amax, int fmt) {
  float t = amax / vmax_f(fmt);
  uint32_t u;
  memcpy(&u, &t, 4);
  u &= 0x7fffffffu;
  if (u == 0) return -127;
  if (u >= 0x7f800000u) return 127;
  uint32_t ex = u >> 23, fr = u & 0x7fffffu;
  int e;
  if (ex != 0) {
    e = (int)ex - 127 + (fr != 0);
  } else {
    int msb = 31 - __builtin_clz(fr);
    e = msb - 149 + ((fr & (fr - 1u)) != 0);
  }
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

int orc_mx_exponent(float amax, int fmt) { return mx_exponent(amax, fmt); }

/* UE8M0 byte -> scale. 0xFF is the NaN code of the format. */
static float ue8m0_to_f32(uint8_t b) {
  if (b == 0xff) return NAN;
  return ldexpf(1.0f, (int)b - 127);
}

/* MX scale-factor tiled layout for the tensor-core block-scaled MMA: the    */
/* row dimension is cut into blocks of 128, the 32-element K-group dimension */
/* into blocks of 4; each 128x4 block occupies 512 bytes, blocks ordered     */
/* row-block-major; inside a block the byte for (row r, group j) sits at     */
/* (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4). This is the public layout  */
/* of 1D block-scaling factors documented for cuBLAS (the 128x4 tile of      */
/* "32 x 16-byte rows").                                                     */
int64_t orc_mx_tiled_offset(int64_t r, int64_t j, int64_t rows, int64_t ngroups) {
  (void)rows;
  int64_t ncb = (ngroups + 3) / 4;
  return ((r / 128) * ncb + j / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

int64_t orc_mx_tiled_bytes(int64_t rows, int64_t ngroups) {
  return ((rows + 127) / 128) * ((ngroups + 3) / 4) * 512;
}

/* ------------------------------------------------------------------ */
/* quantize: x_q = encode(fp32(x * s_inv)) per group, scale stored per group */
/* [Family] "Scaling is what makes FP8 usable" + granularity ladder;         */
/* [Serving] "Quantization Granularity and Scaling Topologies";              */
/* [LowPrec] qdq_e4m3 listing (multiply by 1/s, then satfinite RNE).         */
/* Reading: the pages write round(x / s); the listing multiplies by a        */
/* precomputed 1/s, which is what is done here (fp32 multiply).               */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint16_t *x;
  int64_t rows, cols, ldx;
  int fmt, gran, sf_layout;
  const float *static_scale;
  uint8_t *q;
  int64_t ldq;
  void *scales;
  float tensor_amax_part[256];
  float tensor_s, tensor_s_inv;
} qctx;

static float group_amax(const qctx *c, int64_t r0, int64_t r1, int64_t c0, int64_t c1) {
  float amax = 0.0f;
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t k = c0; k < c1; ++k) {
      float v = fabsf(bf16_to_f32(c->x[r * c->ldx + k]));
      if (v > amax || isnan(v)) amax = v;
    }
  return amax;
}

static void group_encode(const qctx *c, int64_t r0, int64_t r1, int64_t c0, int64_t c1, float s_inv) {
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t k = c0; k < c1; ++k) {
      float v = bf16_to_f32(c->x[r * c->ldx + k]);
      float y = v * s_inv;
      c->q[r * c->ldq + k] = orc_encode_nearest(y, c->fmt);
    }
}

static void q_rows(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  qctx *c = (qctx *)p;
  float *sf = (float *)c->scales;
  uint8_t *sb = (uint8_t *)c->scales;
  for (int64_t r = lo; r < hi; ++r) {
    if (c->gran == ORC_GRAN_TOKEN) {
      float s, si;
      scale_from_amax(group_amax(c, r, r + 1, 0, c->cols), c->fmt, &s, &si);
      sf[r] = s;
      group_encode(c, r, r + 1, 0, c->cols, si);
    } else if (c->gran == ORC_GRAN_TILE_1x128) {
      for (int64_t kb = 0; kb < c->cols / 128; ++kb) {
        float s, si;
        scale_from_amax(group_amax(c, r, r + 1, kb * 128, kb * 128 + 128), c->fmt, &s, &si);
        sf[kb * c->rows + r] = s; /* layout [cols/128][rows], rows contiguous */
        group_encode(c, r, r + 1, kb * 128, kb * 128 + 128, si);
      }
    } else if (c->gran == ORC_GRAN_MX32) {
      int64_t ng = c->cols / 32;
      for (int64_t j = 0; j < ng; ++j) {
        int e = mx_exponent(group_amax(c, r, r + 1, j * 32, j * 32 + 32), c->fmt);
        uint8_t b = (uint8_t)(e + 127);
        if (c->sf_layout == ORC_SF_TILED)
          sb[orc_mx_tiled_offset(r, j, c->rows, ng)] = b;
        else
          sb[r * ng + j] = b;
        group_encode(c, r, r + 1, j * 32, j * 32 + 32, ldexpf(1.0f, -e));
      }
    } else if (c->gran == ORC_GRAN_TENSOR) {
      group_encode(c, r, r + 1, 0, c->cols, c->tensor_s_inv);
    }
  }
}

static void q_blocks(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  qctx *c = (qctx *)p;
  float *sf = (float *)c->scales;
  int64_t nkb = c->cols / 128;
  for (int64_t rb = lo; rb < hi; ++rb) {
    int64_t r0 = rb * 128, r1 = r0 + 128 < c->rows ? r0 + 128 : c->rows;
    for (int64_t kb = 0; kb < nkb; ++kb) {
      float s, si;
      scale_from_amax(group_amax(c, r0, r1, kb * 128, kb * 128 + 128), c->fmt, &s, &si);
      sf[rb * nkb + kb] = s; /* layout [ceil(rows/128)][cols/128] */
      group_encode(c, r0, r1, kb * 128, kb * 128 + 128, si);
    }
  }
}

/* per-channel (one scale per column): "FP8 Serving" guide, Things to try
   (per-channel scales for the KV cache, whose outliers are channel-structured);
   "FP8 Mixed-Precision Serving", FP8 KV Cache section. */
static void q_channel_cols(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  qctx *c = (qctx *)p;
  float *sf = (float *)c->scales;
  for (int64_t k = lo; k < hi; ++k) {
    float s, si;
    scale_from_amax(group_amax(c, 0, c->rows, k, k + 1), c->fmt, &s, &si);
    sf[k] = s;
    group_encode(c, 0, c->rows, k, k + 1, si);
  }
}

static void amax_rows(void *p, int64_t lo, int64_t hi, int tid) {
  qctx *c = (qctx *)p;
  c->tensor_amax_part[tid] = group_amax(c, lo, hi, 0, c->cols);
}

/* Returns 0 on success, -1 on an argument the oracle does not accept. */
int orc_quantize(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int fmt, int gran, int sf_layout,
                 const float *static_scale, uint8_t *q, int64_t ldq, void *scales, int nthreads) {
  if (rows < 0 || cols < 0 || (fmt != ORC_E4M3 && fmt != ORC_E5M2)) return -1;
  if ((gran == ORC_GRAN_TILE_1x128 || gran == ORC_GRAN_BLOCK_128x128) && cols % 128) return -1;
  if (gran == ORC_GRAN_MX32 && cols % 32) return -1;
  if (static_scale && gran != ORC_GRAN_TENSOR) return -1;
  if (gran == ORC_GRAN_CHANNEL && cols % 16) return -1;
  qctx c;
  memset(&c, 0, sizeof c);
  c.x = x;
  c.rows = rows;
  c.cols = cols;
  c.ldx = ldx;
  c.fmt = fmt;
  c.gran = gran;
  c.sf_layout = sf_layout;
  c.static_scale = static_scale;
  c.q = q;
  c.ldq = ldq;
  c.scales = scales;
  switch (gran) {
    case ORC_GRAN_TENSOR: {
      float s, si;
      if (static_scale) {
        /* [Serving] per-tensor static scaling: s is supplied by the caller. */
        s = *static_scale;
        si = 1.0f / s;
        if (s == 0.0f || !isfinite(si)) si = 0.0f;
      } else {
        /* current scaling: the exact amax of the whole tensor first. */
        int nt = resolve_threads(nthreads);
        parallel_for(rows, nt, amax_rows, &c);
        float amax = 0.0f;
        for (int t = 0; t < 256; ++t)
          if (c.tensor_amax_part[t] > amax || isnan(c.tensor_amax_part[t])) amax = c.tensor_amax_part[t];
        scale_from_amax(amax, fmt, &s, &si);
      }
      ((float *)scales)[0] = s;
      c.tensor_s = s;
      c.tensor_s_inv = si;
      parallel_for(rows, nthreads, q_rows, &c);
      return 0;
    }
    case ORC_GRAN_TOKEN:
    case ORC_GRAN_TILE_1x128:
      parallel_for(rows, nthreads, q_rows, &c);
      return 0;
    case ORC_GRAN_MX32:
      if (sf_layout == ORC_SF_TILED) memset(scales, 0, (size_t)orc_mx_tiled_bytes(rows, cols / 32));
      parallel_for(rows, nthreads, q_rows, &c);
      return 0;
    case ORC_GRAN_BLOCK_128x128:
      parallel_for((rows + 127) / 128, nthreads, q_blocks, &c);
      return 0;
    case ORC_GRAN_CHANNEL:
      parallel_for(cols, nthreads, q_channel_cols, &c);
      return 0;
    default:
      return -1;
  }
}

/* Delayed scaling ("FP8 Mixed-Precision Serving", Delayed Scaling vs.
   Just-in-Time Dynamic Scaling: rho = FP8Max / (2^m * max(H)) over an amax
   history H; "Low precision", NVIDIA's taxonomy: per-tensor, delayed).
   Reading: the multiplier rho is formed the way the other scales are:
   s = fp32(fp32(2^m * max(H)) / V_max), rho = s_inv = fp32(1 / s) (0 rule as
   above); an empty or non-finite history (max(H) == 0, inf or NaN) uses s = 1.
   The tensor's own amax then replaces history[slot] (the oldest entry of a
   ring the caller advances one slot per step). */
int orc_quantize_delayed(const uint16_t *x, int64_t rows, int64_t cols, int fmt, const float *history, int hlen,
                         int slot, int margin, uint8_t *q, float *scale_out, float *new_history, int nthreads) {
  if (rows < 0 || cols < 0 || hlen <= 0 || slot < 0 || slot >= hlen || (fmt != ORC_E4M3 && fmt != ORC_E5M2))
    return -1;
  float mh = 0.0f;
  int bad = 0;
  for (int i = 0; i < hlen; ++i) {
    if (!isfinite(history[i])) bad = 1;
    if (history[i] > mh) mh = history[i];
  }
  float s, si;
  if (bad || mh == 0.0f) {
    s = 1.0f;
    si = 1.0f;
  } else {
    float scaled = ldexpf(mh, margin);
    s = scaled / vmax_f(fmt);
    si = 1.0f / s;
    if (s == 0.0f || !isfinite(si)) si = 0.0f;
  }
  qctx c;
  memset(&c, 0, sizeof c);
  c.x = x;
  c.rows = rows;
  c.cols = cols;
  c.ldx = cols;
  c.fmt = fmt;
  c.gran = ORC_GRAN_TENSOR;
  c.q = q;
  c.ldq = cols;
  c.tensor_s = s;
  c.tensor_s_inv = si;
  int nt = resolve_threads(nthreads);
  parallel_for(rows, nt, amax_rows, &c);
  float amax = 0.0f;
  for (int t = 0; t < 256; ++t)
    if (c.tensor_amax_part[t] > amax || isnan(c.tensor_amax_part[t])) amax = c.tensor_amax_part[t];
  parallel_for(rows, nthreads, q_rows, &c);
  *scale_out = s;
  for (int i = 0; i < hlen; ++i) new_history[i] = history[i];
  new_history[slot] = amax;
  return 0;
}

/* ------------------------------------------------------------------ */
/* scale lookup for one element of a quantized [rows x cols] operand        */
/* ------------------------------------------------------------------ */
static double elem_scale(const void *scales, int gran, int sf_layout, int64_t r, int64_t k, int64_t rows,
                         int64_t cols) {
  const float *sf = (const float *)scales;
  const uint8_t *sb = (const uint8_t *)scales;
  switch (gran) {
    case ORC_GRAN_TENSOR:
      return sf[0];
    case ORC_GRAN_TOKEN:
      return sf[r];
    case ORC_GRAN_TILE_1x128:
      return sf[(k / 128) * rows + r];
    case ORC_GRAN_BLOCK_128x128:
      return sf[(r / 128) * (cols / 128) + k / 128];
    case ORC_GRAN_CHANNEL:
      return sf[k];
    case ORC_GRAN_MX32: {
      int64_t ng = cols / 32;
      uint8_t b = sf_layout == ORC_SF_TILED ? sb[orc_mx_tiled_offset(r, k / 32, rows, ng)] : sb[r * ng + k / 32];
      return ue8m0_to_f32(b);
    }
    default:
      return NAN;
  }
}

/* ------------------------------------------------------------------ */
/* dequantize: x_hat = bf16(fp32(decode(q) * s)) ([Family] "x_hat = x_fp8 * s";  */
/* [LowPrec] qdq_e4m3: decode is exact, then one fp32 multiply by s).         */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint8_t *q;
  int64_t rows, cols, ldq;
  int fmt, gran, sf_layout;
  const void *scales;
  uint16_t *out;
  int64_t ldo;
} dqctx;

static void dq_rows(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  dqctx *c = (dqctx *)p;
  for (int64_t r = lo; r < hi; ++r)
    for (int64_t k = 0; k < c->cols; ++k) {
      float d = (float)orc_decode(c->q[r * c->ldq + k], c->fmt);
      float s = (float)elem_scale(c->scales, c->gran, c->sf_layout, r, k, c->rows, c->cols);
      float v = d * s;
      c->out[r * c->ldo + k] = f32_to_bf16_rn(v);
    }
}

int orc_dequantize(const uint8_t *q, int64_t rows, int64_t cols, int64_t ldq, int fmt, int gran, int sf_layout,
                   const void *scales, uint16_t *out, int64_t ldo, int nthreads) {
  if (rows < 0 || cols < 0 || (fmt != ORC_E4M3 && fmt != ORC_E5M2)) return -1;
  dqctx c = {q, rows, cols, ldq, fmt, gran, sf_layout, scales, out, ldo};
  parallel_for(rows, nthreads, dq_rows, &c);
  return 0;
}

/* ------------------------------------------------------------------ */
/* GEMM: ref[m][n] = sum_k x_hat[m][k] * w_hat[n][k] in double, with         */
/* x_hat = decode(q) * s, and bound[m][n] = sum_k |x_hat * w_hat|.          */
/* [Family] "Scaling is what makes FP8 usable": Out = (X_fp8 s_X)(W_fp8 s_W)^T */
/* with fp32 scales; the oracle evaluates the left-hand side directly.      */
/* A = X [M x K] and B = W [N x K], both K-contiguous.                      */
/* rows / cols select the output entries (NULL = all); ref and bound are    */
/* [nrows x ncols].                                                          */
/* ------------------------------------------------------------------ */
typedef struct {
  const uint8_t *a, *b;
  int64_t lda, ldb, M, N, K;
  const void *sa, *sb;
  int a_gran, b_gran, a_sf, b_sf, a_fmt, b_fmt;
  const int64_t *rows, *cols;
  int64_t nrows, ncols;
  const double *ahat; /* [nrows x K] */
  double *ref, *bound;
} gctx;

static void g_deq_a(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  gctx *c = (gctx *)p;
  double *ah = (double *)c->ahat;
  for (int64_t i = lo; i < hi; ++i) {
    int64_t m = c->rows ? c->rows[i] : i;
    for (int64_t k = 0; k < c->K; ++k)
      ah[i * c->K + k] = orc_decode(c->a[m * c->lda + k], c->a_fmt) *
                         elem_scale(c->sa, c->a_gran, c->a_sf, m, k, c->M, c->K);
  }
}

static void g_cols(void *p, int64_t lo, int64_t hi, int tid) {
  (void)tid;
  gctx *c = (gctx *)p;
  double *wh = (double *)malloc(sizeof(double) * (size_t)(c->K > 0 ? c->K : 1));
  for (int64_t j = lo; j < hi; ++j) {
    int64_t n = c->cols ? c->cols[j] : j;
    for (int64_t k = 0; k < c->K; ++k)
      wh[k] = orc_decode(c->b[n * c->ldb + k], c->b_fmt) * elem_scale(c->sb, c->b_gran, c->b_sf, n, k, c->N, c->K);
    for (int64_t i = 0; i < c->nrows; ++i) {
      const double *xh = c->ahat + i * c->K;
      double acc = 0.0, bnd = 0.0;
      for (int64_t k = 0; k < c->K; ++k) {
        double prod = xh[k] * wh[k];
        acc += prod;
        bnd += fabs(prod);
      }
      c->ref[i * c->ncols + j] = acc;
      c->bound[i * c->ncols + j] = bnd;
    }
  }
  free(wh);
}

int orc_gemm(const uint8_t *a, int64_t lda, const void *sa, int a_gran, int a_sf, int a_fmt, const uint8_t *b,
             int64_t ldb, const void *sb, int b_gran, int b_sf, int b_fmt, int64_t M, int64_t N, int64_t K,
             const int64_t *rows, int64_t nrows, const int64_t *cols, int64_t ncols, double *ref, double *bound,
             int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (!rows) nrows = M;
  if (!cols) ncols = N;
  double *ahat = (double *)malloc(sizeof(double) * (size_t)(nrows * K > 0 ? nrows * K : 1));
  if (!ahat) return -2;
  gctx c;
  memset(&c, 0, sizeof c);
  c.a = a;
  c.b = b;
  c.lda = lda;
  c.ldb = ldb;
  c.M = M;
  c.N = N;
  c.K = K;
  c.sa = sa;
  c.sb = sb;
  c.a_gran = a_gran;
  c.b_gran = b_gran;
  c.a_sf = a_sf;
  c.b_sf = b_sf;
  c.a_fmt = a_fmt;
  c.b_fmt = b_fmt;
  c.rows = rows;
  c.cols = cols;
  c.nrows = nrows;
  c.ncols = ncols;
  c.ahat = ahat;
  c.ref = ref;
  c.bound = bound;
  parallel_for(nrows, nthreads, g_deq_a, &c);
  parallel_for(ncols, nthreads, g_cols, &c);
  free(ahat);
  return 0;
}

/* ================================================================== */
/* NVFP4 ([LowPrec] "Low precision: FP8, FP4, and microscaling": NVFP4   */
/* uses blocks of 16 elements, an E4M3 microscale per block and one FP32 */
/* scale per tensor that keeps the microscales inside E4M3's range).     */
/*                                                                        */
/* Readings (the page names FP4 and NVFP4 but prints neither the element */
/* format nor the scale arithmetic):                                      */
/*  - the element format is FP4 E2M1 of the OCP Microscaling spec the     */
/*    page cites: sign, 2 exponent bits (bias 1), 1 mantissa bit; values  */
/*    +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}; no infinity or NaN; encoding rounds */
/*    to nearest, ties to the even code, and saturates at +-6;           */
/*  - tensor scale s_t = fp32(amax_t / (6 * 448)), so that a block holding */
/*    the tensor's amax gets microscale 448 (E4M3's largest value); 1 when */
/*    it comes out 0 or non-finite;                                       */
/*  - block microscale: u = fp32(fp32(amax_b / 6) / s_t), stored as the   */
/*    E4M3 code of u (the FP8 encoder above); s_b = its value (>= 0);     */
/*  - element: S = fp32(s_b * s_t), S_inv = fp32(1 / S) (0 when S is 0 or */
/*    1/S is not finite), q = E2M1(fp32(x * S_inv)), as the 8-bit path     */
/*    multiplies by a precomputed inverse;                                */
/*  - dequantized value: decode(q) * s_b * s_t.                           */
/* ================================================================== */

/* E2M1 code (4 bits) -> value. */
double orc_e2m1_decode(uint32_t c) {
  const int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

/* Nearest representable value by comparison with the midpoints between
   neighbouring magnitudes; a tie takes the code whose mantissa bit is 0. */
uint8_t orc_e2m1_encode_nearest(float xf) {
  const uint8_t sign = signbit(xf) ? 8u : 0u;
  const double a = fabs((double)xf);
  if (isnan(xf)) return 0x7u; /* no NaN in E2M1: not produced for finite inputs */
  uint8_t code = 7;            /* saturate */
  for (uint8_t c = 0; c < 7; ++c) {
    const double lo = orc_e2m1_decode(c), hi = orc_e2m1_decode(c + 1u);
    const double mid = 0.5 * (lo + hi);
    if (a < mid) {
      code = c;
      break;
    }
    if (a == mid) {
      code = (c & 1u) ? (uint8_t)(c + 1u) : c;
      break;
    }
  }
  return (uint8_t)(sign | code);
}

/* The same rounding derived arithmetically: find the binade of |x|, scale the
   significand to one fraction bit, round half to even, then saturate. */
uint8_t orc_e2m1_encode_binade(float xf) {
  const uint8_t sign = signbit(xf) ? 8u : 0u;
  if (isnan(xf)) return 0x7u;
  double a = fabs((double)xf);
  if (a >= 6.0) return (uint8_t)(sign | 7u);
  int e;
  (void)frexp(a, &e);      /* a = f * 2^e, f in [0.5, 1) */
  int ub = e - 1;          /* unbiased exponent of a (a in [2^ub, 2^(ub+1))) */
  if (ub < 0) ub = 0;      /* below 1: the subnormal spacing 0.5 */
  const double step = ldexp(0.5, ub); /* one fraction bit */
  double n = a / step;                /* in [0, 4) units of step */
  double r = floor(n);
  const double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double v = r * step;
  if (v > 6.0) v = 6.0;
  for (uint8_t c = 0; c < 8; ++c)
    if (orc_e2m1_decode(c) == v) return (uint8_t)(sign | c);
  return (uint8_t)(sign | 7u);
}

#define E2M1_MAXT 256
typedef struct {
  uint64_t start;
  int64_t bad[E2M1_MAXT];
  uint64_t first[E2M1_MAXT];
} e2m1_cmp;

static void e2m1_cmp_range(void *p, int64_t lo, int64_t hi, int tid) {
  e2m1_cmp *c = (e2m1_cmp *)p;
  for (int64_t j = lo; j < hi; ++j) {
    const uint32_t u = (uint32_t)(c->start + (uint64_t)j);
    float f;
    memcpy(&f, &u, 4);
    if (isnan(f)) continue;
    if (orc_e2m1_encode_nearest(f) != orc_e2m1_encode_binade(f)) {
      if (!c->bad[tid]) c->first[tid] = c->start + (uint64_t)j;
      ++c->bad[tid];
    }
  }
}

int64_t orc_e2m1_encoders_disagree(uint64_t start, uint64_t count, int nthreads, uint64_t *first_bad) {
  e2m1_cmp *c = (e2m1_cmp *)calloc(1, sizeof(e2m1_cmp));
  if (!c) return -1;
  c->start = start;
  int nt = resolve_threads(nthreads);
  if (nt > E2M1_MAXT) nt = E2M1_MAXT;
  parallel_for((int64_t)count, nt, e2m1_cmp_range, c);
  int64_t bad = 0;
  uint64_t first = 0;
  for (int t = 0; t < E2M1_MAXT; ++t)
    if (c->bad[t]) {
      if (!bad || c->first[t] < first) first = c->first[t];
      bad += c->bad[t];
    }
  free(c);
  if (first_bad) *first_bad = first;
  return bad;
}

/* Compare device-produced E2M1 codes (one per byte) of the fp32 patterns
   start .. start+count-1 with the oracle encoder; NaN inputs are skipped. */
typedef struct {
  uint64_t start;
  const uint8_t *codes;
  int64_t bad[E2M1_MAXT];
  uint64_t first[E2M1_MAXT];
} e2m1_chk;

static void e2m1_chk_range(void *p, int64_t lo, int64_t hi, int tid) {
  e2m1_chk *c = (e2m1_chk *)p;
  for (int64_t j = lo; j < hi; ++j) {
    const uint32_t u = (uint32_t)(c->start + (uint64_t)j);
    float f;
    memcpy(&f, &u, 4);
    if (isnan(f)) continue;
    if ((c->codes[j] & 15u) != orc_e2m1_encode_nearest(f)) {
      if (!c->bad[tid]) c->first[tid] = c->start + (uint64_t)j;
      ++c->bad[tid];
    }
  }
}

int64_t orc_e2m1_check_codes(uint64_t start, uint64_t count, const uint8_t *codes, int nthreads,
                             uint64_t *first_bad) {
  e2m1_chk *c = (e2m1_chk *)calloc(1, sizeof(e2m1_chk));
  if (!c) return -1;
  c->start = start;
  c->codes = codes;
  int nt = resolve_threads(nthreads);
  if (nt > E2M1_MAXT) nt = E2M1_MAXT;
  parallel_for((int64_t)count, nt, e2m1_chk_range, c);
  int64_t bad = 0;
  uint64_t first = 0;
  for (int t = 0; t < E2M1_MAXT; ++t)
    if (c->bad[t]) {
      if (!bad || c->first[t] < first) first = c->first[t];
      bad += c->bad[t];
    }
  free(c);
  if (first_bad) *first_bad = first;
  return bad;
}

float orc_nvfp4_tensor_scale(float amax_t) {
  float s = amax_t / 2688.0f; /* 6 * 448, exact in fp32 */
  if (s == 0.0f || !isfinite(s)) s = 1.0f;
  return s;
}

/* E4M3 code of the block microscale and the element multiplier S_inv. */
static void nvfp4_block_scale(float amax_b, float s_t, uint8_t *code, float *s_b, float *s_inv) {
  const float u = (amax_b / 6.0f) / s_t;
  const uint8_t c = orc_encode_nearest(u, ORC_E4M3);
  const float sb = (float)orc_decode(c, ORC_E4M3);
  const float S = sb * s_t;
  float si = 1.0f / S;
  if (S == 0.0f || !isfinite(si)) si = 0.0f;
  *code = c;
  *s_b = sb;
  *s_inv = si;
}

/* x: bf16 [rows x cols] (row stride ldx elements), cols % 16 == 0.
   q: [rows x cols/2] bytes, element 2i in the low nibble of byte i.
   sf: E4M3 codes, one per 16 elements: linear [rows][cols/16] or the tiled
   128x4 layout of orc_mx_tiled_offset with cols/16 groups.
   *tensor_scale: s_t (computed here from the tensor's amax when
   static_tensor_scale is NULL, else taken from it). */
int orc_quantize_nvfp4(const uint16_t *x, int64_t rows, int64_t cols, int64_t ldx, int sf_layout,
                       const float *static_tensor_scale, uint8_t *q, uint8_t *sf, float *tensor_scale) {
  if (rows < 0 || cols < 0 || cols % 16) return -1;
  float amax_t = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const float v = fabsf(bf16_to_f32(x[r * ldx + c]));
      if (v > amax_t || isnan(v)) amax_t = v;
    }
  const float s_t = static_tensor_scale ? *static_tensor_scale : orc_nvfp4_tensor_scale(amax_t);
  *tensor_scale = s_t;
  const int64_t ng = cols / 16;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < ng; ++g) {
      float amax_b = 0.0f;
      for (int64_t i = 0; i < 16; ++i) {
        const float v = fabsf(bf16_to_f32(x[r * ldx + g * 16 + i]));
        if (v > amax_b) amax_b = v;
      }
      uint8_t code;
      float sb, si;
      nvfp4_block_scale(amax_b, s_t, &code, &sb, &si);
      const int64_t off = sf_layout == ORC_SF_TILED ? orc_mx_tiled_offset(r, g, rows, ng) : r * ng + g;
      sf[off] = code;
      for (int64_t i = 0; i < 16; i += 2) {
        const float a0 = bf16_to_f32(x[r * ldx + g * 16 + i]) * si;
        const float a1 = bf16_to_f32(x[r * ldx + g * 16 + i + 1]) * si;
        q[r * (cols / 2) + (g * 16 + i) / 2] =
            (uint8_t)(orc_e2m1_encode_nearest(a0) | (orc_e2m1_encode_nearest(a1) << 4));
      }
    }
  return 0;
}

static double nvfp4_value(const uint8_t *q, const uint8_t *sf, int sf_layout, float s_t, int64_t r, int64_t k,
                          int64_t rows, int64_t cols) {
  const uint8_t byte = q[r * (cols / 2) + k / 2];
  const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
  const int64_t ng = cols / 16;
  const int64_t off = sf_layout == ORC_SF_TILED ? orc_mx_tiled_offset(r, k / 16, rows, ng) : r * ng + k / 16;
  return orc_e2m1_decode(code) * orc_decode(sf[off], ORC_E4M3) * (double)s_t;
}

/* x_hat = bf16(fp32(decode(q) * fp32(s_b * s_t))). */
int orc_dequantize_nvfp4(const uint8_t *q, const uint8_t *sf, int sf_layout, float s_t, int64_t rows, int64_t cols,
                         uint16_t *out) {
  if (rows < 0 || cols < 0 || cols % 16) return -1;
  const int64_t ng = cols / 16;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t k = 0; k < cols; ++k) {
      const uint8_t byte = q[r * (cols / 2) + k / 2];
      const uint32_t code = (k & 1) ? (byte >> 4) : (byte & 15u);
      const int64_t off = sf_layout == ORC_SF_TILED ? orc_mx_tiled_offset(r, k / 16, rows, ng) : r * ng + k / 16;
      const float S = (float)orc_decode(sf[off], ORC_E4M3) * s_t;
      out[r * cols + k] = f32_to_bf16_rn((float)orc_e2m1_decode(code) * S);
    }
  return 0;
}

/* GEMM over NVFP4 operands: ref = sum_k x_hat * w_hat in double (every
   product of an E2M1 value, an E4M3 microscale and an fp32 tensor scale is
   exact in double), bound = sum_k |x_hat * w_hat|. rows / cols select
   output entries (NULL = all). */
int orc_gemm_nvfp4(const uint8_t *a, const uint8_t *sfa, float sta, const uint8_t *b, const uint8_t *sfb, float stb,
                   int sf_layout, int64_t M, int64_t N, int64_t K, const int64_t *rows, int64_t nrows,
                   const int64_t *cols, int64_t ncols, double *ref, double *bound) {
  if (M < 0 || N < 0 || K < 0 || K % 16) return -1;
  if (!rows) nrows = M;
  if (!cols) ncols = N;
  double *xh = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  double *wh = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)(ncols > 0 ? ncols : 1));
  if (!xh || !wh) {
    free(xh);
    free(wh);
    return -2;
  }
  for (int64_t j = 0; j < ncols; ++j) {
    const int64_t n = cols ? cols[j] : j;
    for (int64_t k = 0; k < K; ++k) wh[j * K + k] = nvfp4_value(b, sfb, sf_layout, stb, n, k, N, K);
  }
  for (int64_t i = 0; i < nrows; ++i) {
    const int64_t m = rows ? rows[i] : i;
    for (int64_t k = 0; k < K; ++k) xh[k] = nvfp4_value(a, sfa, sf_layout, sta, m, k, M, K);
    for (int64_t j = 0; j < ncols; ++j) {
      double acc = 0.0, bnd = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = xh[k] * wh[j * K + k];
        acc += p;
        bnd += fabs(p);
      }
      ref[i * ncols + j] = acc;
      bound[i * ncols + j] = bnd;
    }
  }
  free(xh);
  free(wh);
  return 0;
}
