/*
 * Seeded synthetic-input generators for the hierarchical sparse KV resolve +
 * gather path.
 *
 * This file holds NO arithmetic of the method itself (no resolution, no LRU,
 * no gather).  It only draws the inputs that both the CUDA library and the
 * CPU oracle are fed: KV row payloads, per-step top-k selections, the set of
 * imported-history pages that start optional-resident, and per-step append
 * counts.  The pages describe real GLM-5.3 / DeepSeek-V4.1-Flash traffic
 * ("Adaptive DHiSparse", Evidence section); none of it is available, so these
 * generators stand in for it with the shapes the configurations name.
 *
 * Random numbers: splitmix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014), keyed per purpose so every
 * stream is independent of the order in which streams are drawn.
 * Normals: Box-Muller.  bf16: round-to-nearest-even of the fp32 value.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define DHSW_OK 0
#define DHSW_EINVAL -1
#define DHSW_ENOMEM -2

/* ---------------------------------------------------------------- rng */

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t sm64_next(uint64_t *state) {
  *state += 0x9E3779B97F4A7C15ULL;
  return sm64_mix(*state);
}

/* Uniform double in [0, 1) from the top 53 bits. */
static inline double u01(uint64_t *state) {
  return (double)(sm64_next(state) >> 11) * (1.0 / 9007199254740992.0);
}

/* Uniform integer in [0, n) by 128-bit multiply (Lemire), n >= 1. */
static inline uint64_t below(uint64_t *state, uint64_t n) {
  unsigned __int128 m = (unsigned __int128)sm64_next(state) * n;
  return (uint64_t)(m >> 64);
}

uint64_t dhsw_key(uint64_t seed, uint64_t purpose, uint64_t a, uint64_t b,
                  uint64_t c) {
  uint64_t s = sm64_mix(seed ^ 0x6A09E667F3BCC909ULL);
  s = sm64_mix(s ^ (purpose * 0x9E3779B97F4A7C15ULL));
  s = sm64_mix(s ^ (a + 0x3C6EF372FE94F82BULL));
  s = sm64_mix(s ^ (b + 0xA54FF53A5F1D36F1ULL));
  s = sm64_mix(s ^ (c + 0x510E527FADE682D1ULL));
  return s;
}

enum {
  PURPOSE_PAYLOAD = 1,
  PURPOSE_PERM = 2,
  PURPOSE_SELECT = 3,
  PURPOSE_RESIDENCY = 4,
  PURPOSE_APPEND = 5,
};

/* ---------------------------------------------------------------- bf16 */

uint16_t dhsw_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) /* inf / nan: truncate, keep nan */
    return (uint16_t)((u >> 16) | ((u & 0xFFFFu) ? 0x40u : 0u));
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------- payload */

/* Key of one KV row: (config tag, source, request, row). */
static inline uint64_t row_key(uint64_t seed, uint32_t cfg, uint32_t src,
                               uint32_t req, int64_t row) {
  return dhsw_key(seed, PURPOSE_PAYLOAD, cfg,
                  ((uint64_t)src << 32) | (uint64_t)req, (uint64_t)row);
}

/* Single-precision Box-Muller: one 64-bit draw gives two 24-bit uniforms,
 * u1 in (0, 1] and u2 in [0, 1); the pair of normals is
 * sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2). */
static void payload_row(uint64_t seed, uint32_t cfg, uint32_t src,
                        uint32_t req, int64_t row, int32_t elems,
                        uint16_t *out) {
  uint64_t st = row_key(seed, cfg, src, req, row);
  const float two_pi = 6.28318530717958647692f;
  const float inv24 = 1.0f / 16777216.0f;
  for (int32_t e = 0; e < elems; e += 2) {
    uint64_t x = sm64_next(&st);
    float u1 = (float)((x >> 40) + 1) * inv24;            /* (0, 1] */
    float u2 = (float)((x >> 16) & 0xFFFFFFu) * inv24;    /* [0, 1) */
    float r = sqrtf(-2.0f * logf(u1));
    float a = two_pi * u2;
    out[e] = dhsw_f32_to_bf16(r * cosf(a));
    if (e + 1 < elems) out[e + 1] = dhsw_f32_to_bf16(r * sinf(a));
  }
}

/* One row, single-threaded. */
void dhsw_payload_row(uint64_t seed, uint32_t cfg, uint32_t src, uint32_t req,
                      int64_t row, int32_t elems, uint16_t *out) {
  payload_row(seed, cfg, src, req, row, elems, out);
}

typedef struct {
  uint64_t seed;
  uint32_t cfg;
  const uint32_t *srcs, *reqs;
  int32_t n_pairs;
  int64_t row0, nrows, pair_stride_rows;
  int32_t elems;
  uint16_t *out;
  int64_t begin, end; /* flat (pair, row) range */
} payload_job;

static void *payload_worker(void *arg) {
  payload_job *j = (payload_job *)arg;
  for (int64_t f = j->begin; f < j->end; ++f) {
    int64_t p = f / j->nrows, r = f % j->nrows;
    uint16_t *dst = j->out + (p * j->pair_stride_rows + r) * (int64_t)j->elems;
    payload_row(j->seed, j->cfg, j->srcs[p], j->reqs[p], j->row0 + r, j->elems,
                dst);
  }
  return NULL;
}

/*
 * Rows [row0, row0 + nrows) of every listed (src, req) pair.  Pair p's rows
 * land at out + (p * pair_stride_rows + (row - row0)) * elems.
 */
int dhsw_payload_pairs(uint64_t seed, uint32_t cfg, int32_t n_pairs,
                       const uint32_t *srcs, const uint32_t *reqs,
                       int64_t row0, int64_t nrows, int32_t elems,
                       uint16_t *out, int64_t pair_stride_rows,
                       int32_t nthreads) {
  if (n_pairs < 0 || nrows < 0 || elems <= 0 || pair_stride_rows < nrows)
    return DHSW_EINVAL;
  int64_t total = (int64_t)n_pairs * nrows;
  if (total == 0) return DHSW_OK;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (total < 256) nthreads = 1;
  payload_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = (payload_job){seed, cfg, srcs, reqs, n_pairs, row0, nrows,
                            pair_stride_rows, elems, out,
                            total * t / nthreads, total * (t + 1) / nthreads};
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, payload_worker, &jobs[t]) != 0) break;
    started = t;
  }
  payload_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) payload_worker(&jobs[t]);
  return DHSW_OK;
}

/* ------------------------------------------------- zipf + permutation */

/*
 * Cumulative Zipf(s) weights over ranks 0..n-1 (weight of rank i is
 * (i+1)^-s), normalised so cdf[n-1] == 1.
 */
int dhsw_zipf_cdf(int64_t n, double s, double *cdf) {
  if (n <= 0) return DHSW_EINVAL;
  double acc = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    acc += pow((double)(i + 1), -s);
    cdf[i] = acc;
  }
  for (int64_t i = 0; i < n; ++i) cdf[i] /= acc;
  cdf[n - 1] = 1.0;
  return DHSW_OK;
}

static int64_t zipf_draw(uint64_t *st, const double *cdf, int64_t n) {
  double u = u01(st);
  int64_t lo = 0, hi = n - 1;
  while (lo < hi) { /* first i with cdf[i] > u */
    int64_t mid = lo + (hi - lo) / 2;
    if (cdf[mid] > u) hi = mid; else lo = mid + 1;
  }
  return lo;
}

/* Seeded permutation of [0, n): rank -> history row, per (src, req). */
int dhsw_permutation(uint64_t seed, uint32_t cfg, uint32_t src, uint32_t req,
                     int64_t n, int32_t *out) {
  if (n <= 0) return DHSW_EINVAL;
  for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
  uint64_t st = dhsw_key(seed, PURPOSE_PERM, cfg, src, req);
  for (int64_t i = n - 1; i > 0; --i) {
    int64_t j = (int64_t)below(&st, (uint64_t)(i + 1));
    int32_t t = out[i]; out[i] = out[j]; out[j] = t;
  }
  return DHSW_OK;
}

/* ---------------------------------------------------------------- select */

/* Open-addressing set of non-negative row ids (scratch for one draw). */
typedef struct { int64_t *slots; int64_t cap; } rowset;

static int rowset_init(rowset *s, int64_t want) {
  int64_t cap = 64;
  while (cap < 2 * want + 16) cap <<= 1;
  s->slots = (int64_t *)malloc(sizeof(int64_t) * cap);
  if (!s->slots) return 0;
  for (int64_t i = 0; i < cap; ++i) s->slots[i] = -1;
  s->cap = cap;
  return 1;
}
static int rowset_insert(rowset *s, int64_t v) { /* 1 if newly inserted */
  uint64_t h = sm64_mix((uint64_t)v) & (uint64_t)(s->cap - 1);
  while (s->slots[h] != -1) {
    if (s->slots[h] == v) return 0;
    h = (h + 1) & (uint64_t)(s->cap - 1);
  }
  s->slots[h] = v;
  return 1;
}
static int rowset_has(const rowset *s, int64_t v) {
  uint64_t h = sm64_mix((uint64_t)v) & (uint64_t)(s->cap - 1);
  while (s->slots[h] != -1) {
    if (s->slots[h] == v) return 1;
    h = (h + 1) & (uint64_t)(s->cap - 1);
  }
  return 0;
}

static int cmp_i32(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

/*
 * One top-k selection of `k` distinct rows out of [0, L):
 *   - n_rec = min(round(frac_recent * k), rows of the recency window
 *     [L - min(window, L), L) that are not excluded) rows drawn uniformly
 *     without replacement from that window;
 *   - if rho > 0, each of the previous draw's Zipf rows (prev_z) is kept with
 *     probability rho (unless already taken);
 *   - the rest are distinct Zipf(s) draws over history [0, N): a rank from
 *     the Zipf CDF mapped to a row through the (src, req) permutation,
 *     duplicates rejected.
 * `exclude` (sorted or not, n_exclude rows) may not be chosen.  The k rows
 * are written sorted ascending to out; the Zipf-origin rows (including kept
 * ones) go to out_z (capacity k) and their count to *n_out_z.
 * stream_a/stream_b key the draw (e.g. step and query).
 * Returns DHSW_OK, or DHSW_EINVAL when k rows cannot be found.
 */
int dhsw_select(uint64_t seed, uint32_t cfg, uint32_t src, uint32_t req,
                uint64_t stream_a, uint64_t stream_b, int64_t L, int64_t N,
                int32_t k, int64_t window, double frac_recent,
                const double *cdf, const int32_t *perm, const int32_t *prev_z,
                int32_t n_prev, double rho, const int32_t *exclude,
                int32_t n_exclude, int32_t *out, int32_t *out_z,
                int32_t *n_out_z) {
  if (k < 0 || L < 0 || N < 0 || N > L) return DHSW_EINVAL;
  *n_out_z = 0;
  if (k == 0) return DHSW_OK;
  if ((int64_t)k + n_exclude > L) return DHSW_EINVAL;
  uint64_t st = dhsw_key(seed, PURPOSE_SELECT, cfg,
                         ((uint64_t)src << 32) | (uint64_t)req,
                         (stream_a << 20) ^ stream_b);
  rowset taken;
  if (!rowset_init(&taken, (int64_t)k + n_exclude)) return DHSW_ENOMEM;
  for (int32_t i = 0; i < n_exclude; ++i) rowset_insert(&taken, exclude[i]);
  int32_t n = 0;

  /* recency part: uniform without replacement among free window rows */
  int64_t w = window < L ? window : L;
  int64_t wlo = L - w;
  int64_t *cand = (int64_t *)malloc(sizeof(int64_t) * (size_t)(w > 0 ? w : 1));
  if (!cand) { free(taken.slots); return DHSW_ENOMEM; }
  int64_t nc = 0;
  for (int64_t r = wlo; r < L; ++r)
    if (!rowset_has(&taken, r)) cand[nc++] = r;
  int64_t n_rec = (int64_t)llround(frac_recent * (double)k);
  if (n_rec > nc) n_rec = nc;
  if (n_rec > k) n_rec = k;
  for (int64_t i = 0; i < n_rec; ++i) { /* partial Fisher-Yates */
    int64_t j = i + (int64_t)below(&st, (uint64_t)(nc - i));
    int64_t t = cand[i]; cand[i] = cand[j]; cand[j] = t;
    rowset_insert(&taken, cand[i]);
    out[n++] = (int32_t)cand[i];
  }
  free(cand);

  /* temporal locality: keep previous Zipf rows with probability rho */
  int32_t nz = 0;
  if (rho > 0.0 && prev_z) {
    for (int32_t i = 0; i < n_prev && n < k; ++i) {
      double u = u01(&st);
      if (u < rho && prev_z[i] < L && rowset_insert(&taken, prev_z[i])) {
        out[n++] = prev_z[i];
        out_z[nz++] = prev_z[i];
      }
    }
  }

  /* Zipf part over imported history, duplicates rejected */
  int64_t attempts = 0, limit = 64LL * k + 100000;
  while (n < k && N > 0 && attempts < limit) {
    ++attempts;
    int64_t row = perm[zipf_draw(&st, cdf, N)];
    if (rowset_insert(&taken, row)) {
      out[n++] = (int32_t)row;
      out_z[nz++] = (int32_t)row;
    }
  }
  /* degenerate fallback (tiny histories): lowest free rows, deterministic */
  for (int64_t r = 0; n < k && r < L; ++r)
    if (rowset_insert(&taken, r)) out[n++] = (int32_t)r;
  free(taken.slots);
  if (n < k) return DHSW_EINVAL;
  qsort(out, (size_t)k, sizeof(int32_t), cmp_i32);
  *n_out_z = nz;
  return DHSW_OK;
}

/* ---------------------------------------------------------------- residency */

/*
 * Exactly `count` of the `pages` complete pages of (src, req) marked 1 in
 * mask (uniform without replacement); the rest 0.
 */
int dhsw_residency(uint64_t seed, uint32_t cfg, uint32_t src, uint32_t req,
                   int64_t pages, int64_t count, uint8_t *mask) {
  if (pages < 0 || count < 0 || count > pages) return DHSW_EINVAL;
  memset(mask, 0, (size_t)pages);
  if (count == 0) return DHSW_OK;
  int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)pages);
  if (!idx) return DHSW_ENOMEM;
  for (int64_t i = 0; i < pages; ++i) idx[i] = i;
  uint64_t st = dhsw_key(seed, PURPOSE_RESIDENCY, cfg, src, req);
  for (int64_t i = 0; i < count; ++i) {
    int64_t j = i + (int64_t)below(&st, (uint64_t)(pages - i));
    int64_t t = idx[i]; idx[i] = idx[j]; idx[j] = t;
    mask[idx[i]] = 1;
  }
  free(idx);
  return DHSW_OK;
}

/* ---------------------------------------------------------------- append */

/* Rows appended by request `req` at each of `steps` steps, uniform in
 * [lo, hi]. */
int dhsw_append_counts(uint64_t seed, uint32_t cfg, uint32_t req, int32_t steps,
                       int32_t lo, int32_t hi, int32_t *out) {
  if (steps < 0 || lo < 0 || hi < lo) return DHSW_EINVAL;
  uint64_t st = dhsw_key(seed, PURPOSE_APPEND, cfg, req, 0);
  for (int32_t s = 0; s < steps; ++s)
    out[s] = lo + (int32_t)below(&st, (uint64_t)(hi - lo + 1));
  return DHSW_OK;
}
