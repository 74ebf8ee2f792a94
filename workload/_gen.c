/*
 * Seeded synthetic inputs: standard-normal bf16 rows from a counter-based
 * generator, so that any row can be produced on its own, in any order, by any
 * number of threads, with the same bits on every machine.
 *
 * Definition (the whole generator):
 *   splitmix64(x)   : x += 0x9E3779B97F4A7C15; z = x;
 *                     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
 *                     z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
 *                     return z ^ (z >> 31)            (Steele, Lea & Flood 2014)
 *   row key         : k = splitmix64(seed ^ (domain << 56));
 *                     k = splitmix64(k ^ a); k = splitmix64(k ^ b);
 *                     k = splitmix64(k ^ row)
 *   pair p of a row : h = splitmix64(k + p)
 *                     u1 = ((h >> 40) + 1) / 2^24      in (0, 1]
 *                     u2 = ((h >> 16) & 0xFFFFFF) / 2^24  in [0, 1)
 *                     r = sqrt(-2 ln u1), t = 2 pi u2    (Box & Muller 1958)
 *                     value[2p] = r cos t, value[2p+1] = r sin t
 *   each value is rounded once, from double, to bf16 (round to nearest even).
 *
 * This file holds no arithmetic of the decode path; it only makes inputs.
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static inline uint64_t splitmix64(uint64_t x) {
  uint64_t z = x + 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* double -> bf16 bits, round to nearest even, directly from the double so that
 * no intermediate float rounding happens. Values here are finite and far from
 * the bf16 overflow/underflow range; anything below the normal range flushes
 * to a signed zero. */
static inline uint16_t bf16_from_double(double v) {
  union { double d; uint64_t u; } c;
  c.d = v;
  uint64_t sign = c.u >> 63;
  int64_t e = (int64_t)((c.u >> 52) & 0x7FF);
  uint64_t mant = c.u & 0xFFFFFFFFFFFFFull;
  if (e == 0) return (uint16_t)(sign << 15);
  /* keep 7 mantissa bits: round the low 45 bits away, ties to even */
  uint64_t keep = mant >> 45;
  uint64_t rest = mant & ((1ull << 45) - 1);
  uint64_t half = 1ull << 44;
  if (rest > half || (rest == half && (keep & 1))) keep += 1;
  if (keep == 128) { keep = 0; e += 1; }
  int64_t eb = e - 1023 + 127;
  if (eb <= 0) return (uint16_t)(sign << 15);
  if (eb >= 255) return (uint16_t)((sign << 15) | 0x7F80);
  return (uint16_t)((sign << 15) | ((uint64_t)eb << 7) | keep);
}

static void fill_row(uint16_t* out, int dim, uint64_t seed, uint64_t domain,
                     uint64_t a, uint64_t b, uint64_t row) {
  uint64_t k = splitmix64(seed ^ (domain << 56));
  k = splitmix64(k ^ a);
  k = splitmix64(k ^ b);
  k = splitmix64(k ^ row);
  const double two_pi = 6.283185307179586476925286766559;
  for (int p = 0; 2 * p < dim; ++p) {
    uint64_t h = splitmix64(k + (uint64_t)p);
    double u1 = (double)((h >> 40) + 1) * (1.0 / 16777216.0);
    double u2 = (double)((h >> 16) & 0xFFFFFFull) * (1.0 / 16777216.0);
    double r = sqrt(-2.0 * log(u1));
    double t = two_pi * u2;
    double sn, cs;
    sincos(t, &sn, &cs);
    out[2 * p] = bf16_from_double(r * cs);
    if (2 * p + 1 < dim) out[2 * p + 1] = bf16_from_double(r * sn);
  }
}

typedef struct {
  uint16_t* out;
  int64_t row_stride; /* elements between consecutive rows of out */
  int dim;
  uint64_t seed, domain, a, b;
  int64_t row0, n_rows;
  int64_t first, last; /* [first, last) of the n_rows handled by this worker */
} job_t;

static void* worker(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t i = j->first; i < j->last; ++i)
    fill_row(j->out + i * j->row_stride, j->dim, j->seed, j->domain, j->a, j->b,
             (uint64_t)(j->row0 + i));
  return NULL;
}

/* Fill n_rows rows (row indices row0 .. row0+n_rows-1) of `dim` bf16 values,
 * keyed by (seed, domain, a, b). Returns 0 on success. */
int gen_normal_bf16(uint16_t* out, int64_t row_stride, int dim, uint64_t seed,
                    uint64_t domain, uint64_t a, uint64_t b, int64_t row0,
                    int64_t n_rows, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n_rows < 4096) nthreads = 1;
  pthread_t th[256];
  job_t jobs[256];
  int created[256];
  int64_t per = (n_rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    job_t jb = {out, row_stride, dim, seed, domain, a, b, row0, n_rows,
                t * per < n_rows ? t * per : n_rows,
                (t + 1) * per < n_rows ? (t + 1) * per : n_rows};
    jobs[t] = jb;
    created[t] = 0;
    if (jobs[t].first >= jobs[t].last) continue;
    if (nthreads > 1 && pthread_create(&th[t], NULL, worker, &jobs[t]) == 0)
      created[t] = 1;
    else
      worker(&jobs[t]);
  }
  for (int t = 0; t < nthreads; ++t)
    if (created[t]) pthread_join(th[t], NULL);
  return 0;
}
