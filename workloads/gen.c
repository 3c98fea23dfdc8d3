/*
 * Seeded synthetic input generator for the FP8 lightning indexer and its top-k selector.
 *
 * This file produces INPUTS only: random normals, integers, and the per-row e4m3
 * quantisation that turns a real-valued matrix into e4m3 codes plus an fp32 scale.
 * It contains none of the indexer's arithmetic (no dot products, relu, head sums,
 * scaling of scores, or selection).  Both the CPU oracle and the CUDA path consume
 * what it writes, so neither side can influence the other's inputs.
 *
 * Random numbers: a counter-based generator.  Element i of stream s under seed S is
 *   key   = mix64(S * 0x9E3779B97F4A7C15 + s + 1)
 *   u64   = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 * where mix64 is the SplitMix64 output function (Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014; constants as published by
 * Vigna for splitmix64.c).  Counter-based means every element is a pure function of
 * (seed, stream, index), so the rows can be filled by several threads in any order
 * and the bytes are identical on every machine and thread count.
 *
 * Normals use the Box-Muller transform (Box and Muller, 1958): for element i,
 *   u1 = uniform(2i) in (0,1], u2 = uniform(2i+1) in [0,1),
 *   z  = sqrt(-2 ln u1) * cos(2 pi u2).
 *
 * e4m3 (OCP 8-bit floating point, E4M3FN variant): 1 sign, 4 exponent (bias 7),
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite value 448.
 * Encoding here is round-to-nearest-even with saturation to +-448; it never emits NaN.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define WL_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * WL_GOLDEN + stream + 1ULL);
}

static inline uint64_t draw_u64(uint64_t key, uint64_t i) { return mix64(key + (i + 1ULL) * WL_GOLDEN); }

/* uniform in [0,1) with 53 random bits */
static inline double u01_closed_open(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }
/* uniform in (0,1] with 53 random bits */
static inline double u01_open_closed(uint64_t r) { return (double)((r >> 11) + 1ULL) * 0x1.0p-53; }

static inline double normal_at(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = u01_open_closed(draw_u64(key, 2ULL * i));
  double u2 = u01_closed_open(draw_u64(key, 2ULL * i + 1ULL));
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

uint64_t wl_u64(uint64_t seed, uint64_t stream, uint64_t i) { return draw_u64(stream_key(seed, stream), i); }

/* Round-to-nearest-even, saturating e4m3 encoder (see header comment). */
uint8_t wl_e4m3_encode(double v) {
  uint8_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x80 : 0x00;
  double a = fabs(v);
  if (!(a == a)) return 0x7E; /* NaN input never occurs; map to max rather than emit NaN */
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < 0x1.0p-6) {
    /* subnormal range: value = m * 2^-9, m in 0..7; m == 8 is the smallest normal 2^-6,
       whose code (exponent field 1, mantissa 0) is also 8 */
    double m = rint(a * 512.0); /* default rounding mode: nearest, ties to even */
    return (uint8_t)(sign | (uint8_t)m);
  }
  int e2;
  double f = frexp(a, &e2);     /* a = f * 2^e2, f in [0.5, 1) */
  int ex = e2 - 1;              /* a = (2f) * 2^ex, 2f in [1, 2) */
  double mant = 2.0 * f;
  double q = rint((mant - 1.0) * 8.0);
  if (q >= 8.0) { q = 0.0; ex += 1; }
  int biased = ex + 7;          /* >= 1 here because a >= 2^-6 */
  if (biased > 15 || (biased == 15 && q >= 7.0)) return (uint8_t)(sign | 0x7E);
  return (uint8_t)(sign | (uint8_t)(biased << 3) | (uint8_t)q);
}

/* ---------------------------------------------------------------- threading */

typedef struct {
  int64_t begin, end;
  void (*fn)(void*, int64_t, int64_t);
  void* ctx;
} wl_task;

static void* wl_task_run(void* p) {
  wl_task* t = (wl_task*)p;
  t->fn(t->ctx, t->begin, t->end);
  return NULL;
}

static void wl_parallel_for(int64_t n, int nthreads, void (*fn)(void*, int64_t, int64_t), void* ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 4096 || nthreads == 1) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t th[256];
  wl_task tasks[256];
  int started = 0;
  for (int i = 0; i < nthreads; ++i) {
    tasks[i].begin = n * i / nthreads;
    tasks[i].end = n * (i + 1) / nthreads;
    tasks[i].fn = fn;
    tasks[i].ctx = ctx;
    if (pthread_create(&th[i], NULL, wl_task_run, &tasks[i]) == 0) {
      started = i + 1;
    } else {
      /* could not start a thread: run the rest here */
      for (int j = i; j < nthreads; ++j) {
        tasks[j].begin = n * j / nthreads;
        tasks[j].end = n * (j + 1) / nthreads;
        fn(ctx, tasks[j].begin, tasks[j].end);
      }
      break;
    }
  }
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
}

/* ---------------------------------------------------------------- normals */

typedef struct {
  uint64_t key;
  double std;
  double* out;
} normal_ctx;

static void normal_body(void* p, int64_t b, int64_t e) {
  normal_ctx* c = (normal_ctx*)p;
  for (int64_t i = b; i < e; ++i) c->out[i] = c->std * normal_at(c->key, (uint64_t)i);
}

/* out[i] = std * N(0,1) draw i of (seed, stream), i in [0, n) */
void wl_normal(uint64_t seed, uint64_t stream, int64_t n, double std, double* out, int nthreads) {
  normal_ctx c = {stream_key(seed, stream), std, out};
  wl_parallel_for(n, nthreads, normal_body, &c);
}

/* out[i] = uniform draw i in [0,1) */
void wl_uniform(uint64_t seed, uint64_t stream, int64_t n, double* out) {
  uint64_t key = stream_key(seed, stream);
  for (int64_t i = 0; i < n; ++i) out[i] = u01_closed_open(draw_u64(key, (uint64_t)i));
}

/* out[i] = integer uniform in [lo, hi] (inclusive), by rejection-free multiply-shift on 64 bits.
   The bias of the multiply-shift map is below 2^-32 for ranges below 2^32. */
void wl_uniform_int(uint64_t seed, uint64_t stream, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
  uint64_t key = stream_key(seed, stream);
  uint64_t span = (uint64_t)(hi - lo) + 1ULL;
  for (int64_t i = 0; i < n; ++i) {
    uint64_t r = draw_u64(key, (uint64_t)i) >> 32;
    out[i] = lo + (int64_t)((r * span) >> 32);
  }
}

/* ---------------------------------------------------------------- per-row e4m3 */

typedef struct {
  uint64_t key;
  int64_t cols;
  const double* row_mult;
  uint8_t* codes;
  double* scales;
} rows_ctx;

static void rows_body(void* p, int64_t b, int64_t e) {
  rows_ctx* c = (rows_ctx*)p;
  double* buf = (double*)malloc((size_t)c->cols * sizeof(double));
  if (!buf) return;
  for (int64_t r = b; r < e; ++r) {
    double mult = c->row_mult ? c->row_mult[r] : 1.0;
    double amax = 0.0;
    for (int64_t j = 0; j < c->cols; ++j) {
      double x = mult * normal_at(c->key, (uint64_t)(r * c->cols + j));
      buf[j] = x;
      double a = fabs(x);
      if (a > amax) amax = a;
    }
    double s = amax > 0.0 ? amax / 448.0 : 1.0;
    c->scales[r] = s;
    uint8_t* out = c->codes + r * c->cols;
    for (int64_t j = 0; j < c->cols; ++j) out[j] = wl_e4m3_encode(buf[j] / s);
  }
  free(buf);
}

/* rows x cols matrix of N(0,1) draws (row-major, element r*cols+j is draw r*cols+j of the
   stream), row r multiplied by row_mult[r] (NULL: 1), then quantised per row:
   scales[r] = max_j |x[r,j]| / 448 (1 for an all-zero row), codes[r,j] = e4m3(x[r,j]/scales[r]). */
void wl_normal_e4m3_rows(uint64_t seed, uint64_t stream, int64_t rows, int64_t cols, const double* row_mult,
                         uint8_t* codes, double* scales, int nthreads) {
  rows_ctx c = {stream_key(seed, stream), cols, row_mult, codes, scales};
  wl_parallel_for(rows, nthreads, rows_body, &c);
}

/* codes[i] = e4m3(values[i]) for an array (used to encode small exact integers) */
void wl_encode_e4m3(const double* values, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = wl_e4m3_encode(values[i]);
}
