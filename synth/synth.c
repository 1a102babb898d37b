/*
 * synth.c -- seeded synthetic inputs for the row-wise softmax workloads.
 *
 * Holds none of the softmax arithmetic: only a counter-based random source,
 * the value distributions, and the structural edits (stress entries, a late
 * row maximum, a causal -inf mask).  Both the CUDA path's tests/benchmark and
 * the oracle read the bytes written here.
 *
 * Random source: splitmix64 (S. Vigna's published generator: the n-th output
 * of a stream with state s is mix(s + n * 0x9E3779B97F4A7C15), where mix is
 * the generator's 64-bit finaliser).  Element (r, j) of a matrix drawn with
 * seed `seed` takes outputs 2j+1 and 2j+2 of the stream whose state is
 * mix(seed * golden + r + 1), so any subset of rows can be regenerated alone,
 * in any order, on any number of threads.
 *
 * Values are computed in double, rounded to fp32 (round-to-nearest-even by
 * the C cast), and for bf16 rounded again fp32 -> bf16 (round-to-nearest-
 * even on the bit pattern).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYNTH_F32 0
#define SYNTH_BF16 1
#define SYNTH_F16 2
#define SYNTH_NORMAL 0
#define SYNTH_UNIFORM 1

static const uint64_t kGolden = 0x9E3779B97F4A7C15ull;

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static uint64_t row_state(uint64_t seed, int64_t r) {
  return mix64(seed * kGolden + (uint64_t)r + 1u);
}

/* Output n (n >= 1) of the stream with state s. */
static uint64_t stream_out(uint64_t s, uint64_t n) { return mix64(s + n * kGolden); }

/* A 53-bit uniform in (0, 1]. */
static double unit_open0(uint64_t h) { return ((double)(h >> 11) + 1.0) * 0x1.0p-53; }
/* A 53-bit uniform in [0, 1). */
static double unit_open1(uint64_t h) { return (double)(h >> 11) * 0x1.0p-53; }

static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) { /* inf or nan: keep, quiet nan */
    uint16_t hi = (uint16_t)(u >> 16);
    if (u & 0x007FFFFFu) hi |= 0x0040u;
    return hi;
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static void store_value(void* out, int dtype, int64_t i, double v) {
  float f = (float)v;
  if (dtype == SYNTH_F32) {
    ((float*)out)[i] = f;
  } else if (dtype == SYNTH_F16) {
    _Float16 h = (_Float16)f; /* IEEE binary16, round to nearest even */
    memcpy((uint16_t*)out + i, &h, sizeof h);
  } else {
    ((uint16_t*)out)[i] = f32_to_bf16_rne(f);
  }
}

static double draw(int dist, double p0, double p1, uint64_t s, int64_t j) {
  uint64_t h1 = stream_out(s, 2u * (uint64_t)j + 1u);
  uint64_t h2 = stream_out(s, 2u * (uint64_t)j + 2u);
  if (dist == SYNTH_UNIFORM) return p0 + (p1 - p0) * unit_open1(h1);
  /* Box-Muller: one standard normal from two uniforms */
  double r = sqrt(-2.0 * log(unit_open0(h1)));
  double z = r * cos(6.283185307179586 * unit_open1(h2));
  return p0 + p1 * z;
}

typedef struct {
  void* out;
  int dtype, dist;
  int64_t N, row0, begin, end;
  double p0, p1;
  uint64_t seed;
} fill_job;

static void* fill_worker(void* arg) {
  fill_job* jb = (fill_job*)arg;
  for (int64_t i = jb->begin; i < jb->end; ++i) {
    uint64_t s = row_state(jb->seed, jb->row0 + i);
    for (int64_t j = 0; j < jb->N; ++j)
      store_value(jb->out, jb->dtype, i * jb->N + j, draw(jb->dist, jb->p0, jb->p1, s, j));
  }
  return NULL;
}

/*
 * Rows [row0, row0 + nrows) of an (unbounded) N-column matrix, drawn i.i.d.
 * from dist (SYNTH_NORMAL: mean p0, standard deviation p1; SYNTH_UNIFORM:
 * [p0, p1)), written row-major into out (nrows x N).  Returns 0 or -1.
 */
int synth_fill(void* out, int dtype, int64_t N, int64_t row0, int64_t nrows, int dist,
               double p0, double p1, uint64_t seed, int nthreads) {
  if (!out || N < 1 || nrows < 0 || row0 < 0) return -1;
  if (dtype != SYNTH_F32 && dtype != SYNTH_BF16 && dtype != SYNTH_F16) return -1;
  if (dist != SYNTH_NORMAL && dist != SYNTH_UNIFORM) return -1;
  if (nrows == 0) return 0;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nrows) nthreads = (int)nrows;
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  fill_job* jobs = (fill_job*)calloc((size_t)nthreads, sizeof(fill_job));
  char* started = (char*)calloc((size_t)nthreads, 1);
  if (!tids || !jobs || !started) {
    free(tids);
    free(jobs);
    free(started);
    return -1;
  }
  for (int t = 0; t < nthreads; ++t) {
    fill_job jb = {out, dtype, dist, N, row0, nrows * t / nthreads, nrows * (t + 1) / nthreads,
                   p0, p1, seed};
    jobs[t] = jb;
    if (t > 0 && pthread_create(&tids[t], NULL, fill_worker, &jobs[t]) == 0) started[t] = 1;
  }
  for (int t = 0; t < nthreads; ++t)
    if (!started[t]) fill_worker(&jobs[t]);
  for (int t = 1; t < nthreads; ++t)
    if (started[t]) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  free(started);
  return 0;
}

/* A hash of (seed, a, b) on a stream separate from the value draws. */
static uint64_t side_hash(uint64_t seed, int64_t a, int64_t b) {
  return mix64(mix64(seed ^ 0xD1B54A32D192ED03ull) + (uint64_t)a * kGolden + (uint64_t)b);
}

/*
 * Stress entries: every global row r = row0 + i with r % period == 0 gets the
 * value `hi` at column c1 and `lo` at a different column c2 (both from
 * side_hash).  Needs N >= 2.
 */
int synth_stress_rows(void* out, int dtype, int64_t N, int64_t row0, int64_t nrows, int64_t period,
                      double hi, double lo, uint64_t seed) {
  if (!out || N < 2 || period < 1 || row0 < 0 || nrows < 0) return -1;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = row0 + i;
    if (r % period != 0) continue;
    int64_t c1 = (int64_t)(side_hash(seed, r, 1) % (uint64_t)N);
    int64_t c2 = (int64_t)(side_hash(seed, r, 2) % (uint64_t)(N - 1));
    if (c2 >= c1) ++c2; /* distinct from c1 */
    store_value(out, dtype, i * N + c1, hi);
    store_value(out, dtype, i * N + c2, lo);
  }
  return 0;
}

/*
 * A late row maximum: global row r gets `value` at column
 * p = 3N/4 + side_hash(seed, r) % (N - 3N/4), i.e. in the last quarter.
 */
int synth_late_max(void* out, int dtype, int64_t N, int64_t row0, int64_t nrows, double value,
                   uint64_t seed) {
  if (!out || N < 1 || row0 < 0 || nrows < 0) return -1;
  int64_t lo = 3 * N / 4, span = N - 3 * N / 4;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t r = row0 + i;
    int64_t p = lo + (int64_t)(side_hash(seed, r, 3) % (uint64_t)span);
    store_value(out, dtype, i * N + p, value);
  }
  return 0;
}

/* Position of the late maximum of global row r (for tests). */
int64_t synth_late_max_col(int64_t N, int64_t r, uint64_t seed) {
  return 3 * N / 4 + (int64_t)(side_hash(seed, r, 3) % (uint64_t)(N - 3 * N / 4));
}

/*
 * Causal mask: global row r is query q = r % q_len; columns j > q are set
 * to -inf.
 */
int synth_causal_mask(void* out, int dtype, int64_t N, int64_t row0, int64_t nrows, int64_t q_len) {
  if (!out || N < 1 || q_len < 1 || row0 < 0 || nrows < 0) return -1;
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t q = (row0 + i) % q_len;
    for (int64_t j = q + 1; j < N; ++j) store_value(out, dtype, i * N + j, -INFINITY);
  }
  return 0;
}
