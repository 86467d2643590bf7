/*
 * CPU ORACLE for hierarchical sparse KV resolution + gather.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library; both are fed by the seeded input
 * generators alone.
 *
 * It is a plain, slow, literal statement of what "Adaptive DHiSparse:
 * Speculative Decoding over a Load-Adaptive KV Hierarchy" describes under
 * "How it works":
 *   - Memory split: every (request, KV source) pair owns B hot-cache rows, its
 *     tail ring and its metadata, none of them lent out; whole pages of
 *     imported history may occupy optional capacity that can be taken back,
 *     as long as required, optional and the admission reserve together fit
 *     the pool.
 *   - Reclamation: whole requests' optional pages are taken in reclaim order
 *     until the deficit is covered, otherwise the admission waits.
 *   - Resolution: each selected row is looked for in three places in turn,
 *     stopping at the first that holds it -- (1) the tail ring, then the map
 *     of optional pages resident on the GPU; (2) the B hot-cache tags, the
 *     least recently used slots giving way; (3) its pinned host copy,
 *     fetched into the hot cache.
 *   - Speculative state: the queries of a verify block fetch a missing row
 *     once between them; a drafter retains only the rows its window covers,
 *     stored as a ring (a window source: the tail ring is its only storage).
 *   - Model-specific reuse: a Reuse layer takes over the location vector of
 *     the layer before it (here: a gather of an existing location vector, no
 *     resolution).
 *   - Limits: decode rows are served the hot-cache way.
 *
 * Readings where the pages are silent (each restated beside the code):
 *   tail = the most recent T rows [L-T, L) held in a ring at row mod T,
 *   including imported rows at admission; tail is consulted before the
 *   optional map; step-1 hits do not touch LRU state; LRU = per-slot
 *   last-use step stamps, empty slots (tag -1, stamp 0) first, smallest
 *   (stamp, slot) evicted, misses handled in ascending row order, slots hit
 *   or filled in this step protected; a step that needs more victims than
 *   unprotected slots fails with EBUDGET and changes nothing (its step-1
 *   rows keep their locations, every other entry has none); duplicates in
 *   a selection share one location and count once; a verify block is one
 *   step; optional slots are allocated lowest-free-first, pages ascending.
 *
 * Location encoding: (tier << 30) | index; tier 0 = tail (index
 * pair*T + row mod T), 1 = optional (index slot*page_rows + row mod
 * page_rows), 2 = hot (index pair*B + slot); 0xFFFFFFFF = no location;
 * 0xFFFFFFFE = past the end of a union location list (union staging).
 * Counters per resolve: entries, unique, tail, optional, hot, host,
 * scan_max (probes of the longest hot-cache scan), evicted (victims that
 * held a row).
 *
 * Calls on different (request, source) pairs touch disjoint state and may
 * run on different threads at once; admission, reclaim and release may not
 * overlap any other call.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL -1
#define ORC_ENOMEM -2
#define ORC_EWOULDWAIT -3
#define ORC_EBUDGET -4
#define ORC_ERANGE -5
#define ORC_ESTATE -8

#define ORC_TIER_TAIL 0u
#define ORC_TIER_OPT 1u
#define ORC_TIER_HOT 2u
#define ORC_NO_LOC 0xFFFFFFFFu
#define ORC_END_LOC 0xFFFFFFFEu /* past the end of a union location list */

typedef struct {
  int admitted;
  int tracked;        /* holds row bytes (else metadata only) */
  int window;         /* a window source: the tail ring is its only storage */
  int64_t N;          /* imported rows */
  int64_t L;          /* current length */
  int32_t *page_slot; /* [pages_max]: optional-pool slot, -1 = not ready */
  int32_t *tags;      /* [B]: row held by each hot slot, -1 = empty */
  uint32_t *stamps;   /* [B]: step of last use, 0 = never */
  uint16_t *host;     /* [max_rows][E]: this source's pinned-host copy */
  uint16_t *tail;     /* [T][E] */
  uint16_t *hot;      /* [B][E] */
  /* resident-first admission from device rows: the imported rows as the
   * device holds them (what a ready optional page contains); NULL when the
   * source was admitted from its host copy */
  uint16_t *imported;
  uint8_t *backed;    /* [pages_max]: 1 = the host copy of the page is valid */
  uint64_t *pend;     /* [pages_max]: backup order of a pending page, 0 = none */
} orc_source;

typedef struct {
  int32_t R, S, T, B, E, PR;
  int32_t rr;         /* refill cursor: the next request visited */
  uint64_t bseq;      /* pages put in backup order so far */
  int64_t max_rows, pages_max, capacity, reserve, used, first_free;
  int32_t *slot_pair; /* [capacity]: owning pair, -1 = free */
  int32_t *slot_page; /* [capacity]: page of the owner */
  orc_source *src;    /* [R*S] */
} orc_pool;

static void reset_source_state(const orc_pool *p, orc_source *s) {
  for (int32_t j = 0; j < p->B; ++j) { s->tags[j] = -1; s->stamps[j] = 0; }
  for (int64_t q = 0; q < p->pages_max; ++q) {
    s->page_slot[q] = -1;
    s->backed[q] = 1;
    s->pend[q] = 0;
  }
  s->admitted = 0; s->tracked = 0; s->window = 0; s->N = 0; s->L = 0;
  free(s->host); free(s->tail); free(s->hot); free(s->imported);
  s->host = s->tail = s->hot = s->imported = NULL;
}

void orc_pool_free(orc_pool *p) {
  if (!p) return;
  if (p->src) {
    for (int64_t i = 0; i < (int64_t)p->R * p->S; ++i) {
      orc_source *s = &p->src[i];
      free(s->page_slot); free(s->tags); free(s->stamps);
      free(s->host); free(s->tail); free(s->hot); free(s->imported);
      free(s->backed); free(s->pend);
    }
  }
  free(p->src); free(p->slot_pair); free(p->slot_page); free(p);
}

orc_pool *orc_pool_new(int32_t R, int32_t S, int32_t T, int32_t B, int32_t E,
                       int32_t PR, int64_t max_rows, int64_t capacity_pages,
                       int64_t reserve_pages) {
  if (R <= 0 || S <= 0 || T <= 0 || B <= 0 || E <= 0 || PR <= 0 ||
      max_rows <= 0 || capacity_pages < 0 || reserve_pages < 0 ||
      reserve_pages > capacity_pages)
    return NULL;
  orc_pool *p = (orc_pool *)calloc(1, sizeof(orc_pool));
  if (!p) return NULL;
  p->R = R; p->S = S; p->T = T; p->B = B; p->E = E; p->PR = PR;
  p->max_rows = max_rows;
  p->pages_max = (max_rows + PR - 1) / PR;
  p->capacity = capacity_pages; p->reserve = reserve_pages;
  p->slot_pair = (int32_t *)malloc(sizeof(int32_t) * (size_t)(capacity_pages + 1));
  p->slot_page = (int32_t *)malloc(sizeof(int32_t) * (size_t)(capacity_pages + 1));
  p->src = (orc_source *)calloc((size_t)R * S, sizeof(orc_source));
  if (!p->slot_pair || !p->slot_page || !p->src) { orc_pool_free(p); return NULL; }
  for (int64_t i = 0; i < capacity_pages; ++i) { p->slot_pair[i] = -1; p->slot_page[i] = -1; }
  for (int64_t i = 0; i < (int64_t)R * S; ++i) {
    orc_source *s = &p->src[i];
    s->page_slot = (int32_t *)malloc(sizeof(int32_t) * (size_t)p->pages_max);
    s->tags = (int32_t *)malloc(sizeof(int32_t) * (size_t)B);
    s->stamps = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)B);
    s->backed = (uint8_t *)malloc((size_t)p->pages_max);
    s->pend = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)p->pages_max);
    if (!s->page_slot || !s->tags || !s->stamps || !s->backed || !s->pend) {
      orc_pool_free(p);
      return NULL;
    }
    reset_source_state(p, s);
  }
  return p;
}

static orc_source *get_src(orc_pool *p, int32_t r, int32_t s) {
  if (!p || r < 0 || r >= p->R || s < 0 || s >= p->S) return NULL;
  return &p->src[(int64_t)r * p->S + s];
}

int64_t orc_pool_used(const orc_pool *p) { return p ? p->used : -1; }

/* ------------------------------------------------------------ admission */

static int64_t lowest_free_slot(orc_pool *p) {
  /* every slot below first_free is occupied */
  for (int64_t i = p->first_free; i < p->capacity; ++i)
    if (p->slot_pair[i] < 0) { p->first_free = i; return i; }
  return -1;
}

static void free_slot(orc_pool *p, int64_t slot) {
  p->slot_pair[slot] = -1; p->slot_page[slot] = -1;
  p->used -= 1;
  if (slot < p->first_free) p->first_free = slot;
}

/*
 * Admit (r, s) with N imported rows.  Resident-first: every complete page
 * marked in `mask` (NULL = all complete pages) takes an optional slot,
 * lowest free slot first, pages ascending.  If required + optional +
 * admission reserve would exceed capacity the call changes nothing, stores
 * the missing page count in *deficit and returns ORC_EWOULDWAIT (the
 * admission waits).  `host_rows` (N rows) are this source's host copy; NULL
 * keeps metadata only.
 */
int orc_admit(orc_pool *p, int32_t r, int32_t s, const uint16_t *host_rows,
              int64_t N, const uint8_t *mask, int64_t *deficit) {
  orc_source *src = get_src(p, r, s);
  if (deficit) *deficit = 0;
  if (!src || N < 0 || N > p->max_rows) return ORC_EINVAL;
  if (src->admitted) return ORC_ESTATE;
  int64_t complete = N / p->PR, want = 0;
  for (int64_t q = 0; q < complete; ++q) want += (!mask || mask[q]) ? 1 : 0;
  if (p->used + want > p->capacity - p->reserve) {
    if (deficit) *deficit = p->used + want - (p->capacity - p->reserve);
    return ORC_EWOULDWAIT;
  }
  int64_t pair = (int64_t)r * p->S + s;
  if (host_rows) {
    size_t E = (size_t)p->E;
    src->host = (uint16_t *)calloc((size_t)p->max_rows * E, 2);
    src->tail = (uint16_t *)calloc((size_t)p->T * E, 2);
    src->hot = (uint16_t *)calloc((size_t)p->B * E, 2);
    if (!src->host || !src->tail || !src->hot) {
      free(src->host); free(src->tail); free(src->hot);
      src->host = src->tail = src->hot = NULL;
      return ORC_ENOMEM;
    }
    memcpy(src->host, host_rows, (size_t)N * E * 2);
    int64_t lo = N - p->T > 0 ? N - p->T : 0;
    for (int64_t row = lo; row < N; ++row) /* tail holds [N-T, N) */
      memcpy(src->tail + (size_t)(row % p->T) * E, src->host + (size_t)row * E, E * 2);
    src->tracked = 1;
  }
  for (int64_t q = 0; q < complete; ++q) {
    if (mask && !mask[q]) continue;
    int64_t slot = lowest_free_slot(p);
    p->slot_pair[slot] = (int32_t)pair;
    p->slot_page[slot] = (int32_t)q;
    p->used += 1;
    src->page_slot[q] = (int32_t)slot;
  }
  src->N = N; src->L = N; src->admitted = 1;
  return ORC_OK;
}

int orc_release(orc_pool *p, int32_t r);

#define ORC_POISON 0xDEADu /* host rows whose backup has not happened yet */

/*
 * Resident-first admission of rows that are on the device ("Resident-first
 * admission": while HBM has room, an arriving request's imported history
 * stays on the GPU and its host backup is put off).  `rows` (N rows, NULL = metadata
 * only) are the imported rows as the device holds them.  Pages are chosen
 * and the capacity rule applied exactly as in orc_admit.  Every complete
 * page marked in `mask` becomes a ready optional page whose host backup is
 * deferred: it joins the backup order and its host rows are not valid yet.
 * Every other imported row (pages left out, the incomplete last page) can
 * only be served from host memory, so it is copied to the host now.
 */
int orc_admit_device(orc_pool *p, int32_t r, int32_t s, const uint16_t *rows,
                     int64_t N, const uint8_t *mask, int64_t *deficit) {
  orc_source *src = get_src(p, r, s);
  if (deficit) *deficit = 0;
  if (!src || N < 0 || N > p->max_rows) return ORC_EINVAL;
  if (src->admitted) return ORC_ESTATE;
  size_t E = (size_t)p->E;
  uint16_t *imported = NULL;
  if (rows) {
    imported = (uint16_t *)malloc((size_t)N * E * 2 + 2);
    if (!imported) return ORC_ENOMEM;
    memcpy(imported, rows, (size_t)N * E * 2);
  }
  int rc = orc_admit(p, r, s, rows, N, mask, deficit);
  if (rc != ORC_OK) {
    free(imported);
    return rc;
  }
  src->imported = imported;
  for (int64_t q = 0; q < N / p->PR; ++q) {
    if (src->page_slot[q] < 0) continue;
    src->backed[q] = 0;
    src->pend[q] = ++p->bseq;
    if (src->host)
      for (size_t i = 0; i < (size_t)p->PR * E; ++i)
        src->host[(size_t)q * p->PR * E + i] = ORC_POISON;
  }
  return ORC_OK;
}

/* Copy one pending page's rows from the device copy to the host copy. */
static void backup_page(orc_source *src, const orc_pool *p, int64_t q) {
  if (src->host && src->imported) {
    size_t n = (size_t)p->PR * p->E;
    memcpy(src->host + (size_t)q * n, src->imported + (size_t)q * n, n * 2);
  }
  src->backed[q] = 1;
  src->pend[q] = 0;
}

/*
 * Back up at most max_pages pending pages, in backup order (admission order,
 * pages ascending); *done = pages backed up.
 */
int orc_backup(orc_pool *p, int64_t max_pages, int64_t *done) {
  if (done) *done = 0;
  if (!p || max_pages < 0) return ORC_EINVAL;
  int64_t n = 0;
  while (n < max_pages) {
    orc_source *best = NULL;
    int64_t best_q = -1;
    for (int64_t i = 0; i < (int64_t)p->R * p->S; ++i) {
      orc_source *src = &p->src[i];
      for (int64_t q = 0; q < p->pages_max; ++q)
        if (src->pend[q] && (!best || src->pend[q] < best->pend[best_q])) {
          best = src;
          best_q = q;
        }
    }
    if (!best) break;
    backup_page(best, p, best_q);
    n++;
  }
  if (done) *done = n;
  return ORC_OK;
}

int64_t orc_pending_backup(const orc_pool *p) {
  int64_t n = 0;
  for (int64_t i = 0; p && i < (int64_t)p->R * p->S; ++i)
    for (int64_t q = 0; q < p->pages_max; ++q) n += p->src[i].pend[q] != 0;
  return n;
}

/*
 * Bounded round-robin refill ("Reclamation and refill": refill uses bounded
 * round-robin).  Requests are visited cyclically from the cursor; a visit
 * to a request with a complete imported page that is not optional-resident
 * makes its lowest (source, page) such page resident again (lowest free
 * slot; the bytes come from the host copy, which such a page always has).
 * It stops after max_pages pages, when the capacity rule (used <= capacity
 * - reserve) leaves no room, or when a whole round of visits found nothing.
 * The cursor keeps the next request to visit.  *filled = pages refilled.
 */
int orc_refill(orc_pool *p, int64_t max_pages, int64_t *filled) {
  if (filled) *filled = 0;
  if (!p || max_pages < 0) return ORC_EINVAL;
  int64_t n = 0, idle = 0;
  int32_t r = p->rr;
  while (n < max_pages && p->used < p->capacity - p->reserve && idle < p->R) {
    int found = 0;
    for (int32_t s = 0; s < p->S && !found; ++s) {
      orc_source *src = &p->src[(int64_t)r * p->S + s];
      if (!src->admitted) continue;
      for (int64_t q = 0; q < src->N / p->PR && !found; ++q) {
        if (src->page_slot[q] >= 0) continue;
        int64_t slot = lowest_free_slot(p);
        p->slot_pair[slot] = (int32_t)((int64_t)r * p->S + s);
        p->slot_page[slot] = (int32_t)q;
        p->used += 1;
        src->page_slot[q] = (int32_t)slot;
        found = 1;
      }
    }
    if (found) { n++; idle = 0; } else { idle++; }
    r = (r + 1) % p->R;
  }
  p->rr = r;
  if (filled) *filled = n;
  return ORC_OK;
}

static int64_t request_pages(const orc_pool *p, int32_t r) {
  int64_t n = 0;
  for (int32_t s = 0; s < p->S; ++s) {
    const orc_source *src = &p->src[(int64_t)r * p->S + s];
    for (int64_t q = 0; q < p->pages_max; ++q) n += src->page_slot[q] >= 0;
  }
  return n;
}

/*
 * Walk `order` and take whole requests' optional pages (all their sources)
 * until `deficit` pages are freed.  If the listed requests cannot cover the
 * deficit nothing is taken and ORC_EWOULDWAIT is returned.
 */
int orc_reclaim(orc_pool *p, const int32_t *order, int32_t n, int64_t deficit,
                int64_t *freed) {
  if (freed) *freed = 0;
  if (!p || n < 0 || deficit < 0 || (n > 0 && !order)) return ORC_EINVAL;
  for (int32_t i = 0; i < n; ++i)
    if (order[i] < 0 || order[i] >= p->R) return ORC_EINVAL;
  /* can the listed requests cover it?  (each request counted once) */
  int64_t avail = 0;
  for (int32_t i = 0; i < n; ++i) {
    int dup = 0;
    for (int32_t j = 0; j < i; ++j) dup |= order[j] == order[i];
    if (!dup) avail += request_pages(p, order[i]);
  }
  if (avail < deficit) return ORC_EWOULDWAIT;
  int64_t got = 0;
  for (int32_t i = 0; i < n && got < deficit; ++i) {
    int32_t r = order[i];
    for (int32_t s = 0; s < p->S; ++s) {
      orc_source *src = &p->src[(int64_t)r * p->S + s];
      for (int64_t q = 0; q < p->pages_max; ++q) {
        if (src->page_slot[q] < 0) continue;
        /* a page is freed only after its host backup is complete */
        if (!src->backed[q]) backup_page(src, p, q);
        free_slot(p, src->page_slot[q]);
        src->page_slot[q] = -1;
        got += 1;
      }
    }
  }
  if (freed) *freed = got;
  return ORC_OK;
}

/* Release every source of request r: pages freed, state back to empty. */
int orc_release(orc_pool *p, int32_t r) {
  if (!p || r < 0 || r >= p->R) return ORC_EINVAL;
  for (int32_t s = 0; s < p->S; ++s) {
    orc_source *src = &p->src[(int64_t)r * p->S + s];
    for (int64_t q = 0; q < p->pages_max; ++q)
      if (src->page_slot[q] >= 0) free_slot(p, src->page_slot[q]);
    reset_source_state(p, src);
  }
  return ORC_OK;
}

/*
 * Admit (r, s) as a window source ("Speculative state": a drafter retains
 * only the rows its window covers, stored as a ring).  The ring of T rows is all the
 * source has: no host copy, no optional pages (it takes no capacity), and its
 * rows never enter the hot cache.  A window of N rows holds rows
 * [N - m, N), m = min(N, T), at ring slots row mod T; `rows` gives those m
 * rows in order (NULL = metadata only).  L = N; N counts no imported pages.
 */
int orc_admit_window(orc_pool *p, int32_t r, int32_t s, const uint16_t *rows, int64_t N) {
  orc_source *src = get_src(p, r, s);
  if (!src || N < 0 || N > p->max_rows) return ORC_EINVAL;
  if (src->admitted) return ORC_ESTATE;
  if (rows) {
    size_t E = (size_t)p->E;
    src->tail = (uint16_t *)calloc((size_t)p->T * E, 2);
    src->hot = (uint16_t *)calloc((size_t)p->B * E, 2);
    if (!src->tail || !src->hot) {
      free(src->tail); free(src->hot);
      src->tail = src->hot = NULL;
      return ORC_ENOMEM;
    }
    int64_t m = N < p->T ? N : p->T;
    for (int64_t j = 0; j < m; ++j) {
      int64_t row = N - m + j;
      memcpy(src->tail + (size_t)(row % p->T) * E, rows + (size_t)j * E, E * 2);
    }
    src->tracked = 1;
  }
  src->window = 1;
  src->N = 0; src->L = N; src->admitted = 1;
  return ORC_OK;
}

/* ------------------------------------------------------------ append */

/*
 * Append `count` decode rows to (r, s): row L+j goes to tail slot
 * (L+j) mod T and is written through to the host copy, so every row keeps
 * a host copy once it leaves the tail.  A window source has no host copy:
 * the row it overwrites leaves the window for good.  count <= T.
 */
int orc_append(orc_pool *p, int32_t r, int32_t s, int32_t count,
               const uint16_t *rows) {
  orc_source *src = get_src(p, r, s);
  if (!src || count < 0 || count > p->T) return ORC_EINVAL;
  if (!src->admitted) return ORC_ESTATE;
  if (src->L + count > p->max_rows) return ORC_EINVAL;
  if (src->tracked) {
    if (count > 0 && !rows) return ORC_EINVAL;
    size_t E = (size_t)p->E;
    for (int32_t j = 0; j < count; ++j) {
      int64_t row = src->L + j;
      memcpy(src->tail + (size_t)(row % p->T) * E, rows + (size_t)j * E, E * 2);
      if (!src->window) memcpy(src->host + (size_t)row * E, rows + (size_t)j * E, E * 2);
    }
  }
  src->L += count;
  return ORC_OK;
}

/* ------------------------------------------------------------ resolve */

static int cmp_i32(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

static int64_t find_sorted(const int32_t *u, int64_t n, int32_t v) {
  int64_t lo = 0, hi = n - 1;
  while (lo <= hi) {
    int64_t mid = lo + (hi - lo) / 2;
    if (u[mid] == v) return mid;
    if (u[mid] < v) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

/*
 * Step 1 of Resolution for one row of (r, s): the mutable tail holds rows
 * [L-T, L) at ring slot row mod T; else the ready optional-history map
 * (complete imported pages only, "Memory split").  The row's location, or
 * ORC_NO_LOC when step 1 does not hold it (or the row is outside [0, L)).
 */
static uint32_t step1_location(const orc_pool *p, const orc_source *src,
                               int64_t pair, int64_t row) {
  const int64_t L = src->L, N = src->N, T = p->T, PR = p->PR;
  if (row < 0 || row >= L) return ORC_NO_LOC;
  if (row >= L - T) return (ORC_TIER_TAIL << 30) | (uint32_t)(pair * T + row % T);
  int64_t page = row / PR;
  if ((page + 1) * PR <= N && src->page_slot[page] >= 0)
    return (ORC_TIER_OPT << 30) |
           (uint32_t)((int64_t)src->page_slot[page] * PR + row % PR);
  return ORC_NO_LOC;
}

/*
 * Resolve the Q x k selection `sel` of (r, s) at `step` (>= 1) into `loc`
 * (Q*k) and `counters` (8).  A window source holds only rows [L-T, L): any
 * other row is out of its range.  On ORC_ERANGE (a row outside [0, L), or
 * outside a window source's window) or
 * ORC_EBUDGET (more misses than unprotected hot slots) nothing changes and
 * every counter is 0; step 1 reads no state that resolution changes, so the
 * entries it resolves keep their locations and every other entry is
 * ORC_NO_LOC.
 */
int orc_resolve(orc_pool *p, uint32_t step, int32_t r, int32_t s, int32_t Q,
                int32_t k, const int32_t *sel, uint32_t *loc,
                uint32_t *counters) {
  orc_source *src = get_src(p, r, s);
  if (!src || step == 0 || Q < 0 || k < 0) return ORC_EINVAL;
  if (!src->admitted) return ORC_ESTATE;
  int64_t n = (int64_t)Q * k;
  const int64_t pair = (int64_t)r * p->S + s;
  const int64_t L = src->L, B = p->B;
  for (int c = 0; c < 8; ++c) counters[c] = 0;
  /* lowest row the source can serve: a window source only has its ring */
  const int64_t lo = src->window && L > p->T ? L - p->T : 0;
  for (int64_t e = 0; e < n; ++e)
    if ((int64_t)sel[e] < lo || (int64_t)sel[e] >= L) {
      for (int64_t f = 0; f < n; ++f) loc[f] = step1_location(p, src, pair, sel[f]);
      return ORC_ERANGE;
    }

  /* all verify queries together: sorted union of the selected rows */
  int32_t *U = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  uint32_t *where = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(n + 1));
  uint8_t *miss = (uint8_t *)calloc((size_t)(n + 1), 1);
  uint32_t *st = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)B);
  if (!U || !where || !miss || !st) {
    free(U); free(where); free(miss); free(st);
    return ORC_ENOMEM;
  }
  memcpy(U, sel, sizeof(int32_t) * (size_t)n);
  qsort(U, (size_t)n, sizeof(int32_t), cmp_i32);
  int64_t nu = 0;
  for (int64_t e = 0; e < n; ++e)
    if (nu == 0 || U[nu - 1] != U[e]) U[nu++] = U[e];
  memcpy(st, src->stamps, sizeof(uint32_t) * (size_t)B);

  uint32_t c_tail = 0, c_opt = 0, c_hot = 0, c_host = 0, scan_max = 0, evicted = 0;
  int64_t n_miss = 0;
  for (int64_t u = 0; u < nu; ++u) {
    int64_t row = U[u];
    /* step 1: the tail, then the ready optional-history map */
    uint32_t l1 = step1_location(p, src, pair, row);
    if (l1 != ORC_NO_LOC) {
      where[u] = l1;
      if ((l1 >> 30) == ORC_TIER_TAIL) c_tail++; else c_opt++;
      continue;
    }
    /* step 2: the B hot-cache tags, in slot order */
    int64_t j = 0;
    while (j < B && src->tags[j] != row) ++j;
    if (j < B) {
      where[u] = (ORC_TIER_HOT << 30) | (uint32_t)(pair * B + j);
      st[j] = step;
      c_hot++;
      if ((uint32_t)(j + 1) > scan_max) scan_max = (uint32_t)(j + 1);
    } else {
      miss[u] = 1;
      n_miss++;
      scan_max = (uint32_t)B;
    }
  }

  /* step 3 needs one unprotected victim per missing row */
  int64_t avail = 0;
  for (int64_t j = 0; j < B; ++j) avail += st[j] != step;
  if (n_miss > avail) {
    for (int64_t e = 0; e < n; ++e) loc[e] = step1_location(p, src, pair, sel[e]);
    free(U); free(where); free(miss); free(st);
    return ORC_EBUDGET;
  }
  /* step 3: missing rows in ascending order, each into the least recently
   * used unprotected slot (smallest stamp, then lowest slot) */
  for (int64_t u = 0; u < nu; ++u) {
    if (!miss[u]) continue;
    int64_t best = -1;
    for (int64_t j = 0; j < B; ++j) {
      if (st[j] == step) continue;
      if (best < 0 || st[j] < st[best]) best = j;
    }
    if (src->tags[best] != -1) evicted++;
    src->tags[best] = U[u];
    st[best] = step;
    if (src->tracked)
      memcpy(src->hot + (size_t)best * p->E, src->host + (size_t)U[u] * p->E,
             (size_t)p->E * 2);
    where[u] = (ORC_TIER_HOT << 30) | (uint32_t)(pair * B + best);
    c_host++;
  }
  memcpy(src->stamps, st, sizeof(uint32_t) * (size_t)B);

  /* location vector: every entry takes its row's location */
  for (int64_t e = 0; e < n; ++e) loc[e] = where[find_sorted(U, nu, sel[e])];
  counters[0] = (uint32_t)n;
  counters[1] = (uint32_t)nu;
  counters[2] = c_tail;
  counters[3] = c_opt;
  counters[4] = c_hot;
  counters[5] = c_host;
  counters[6] = scan_max;
  counters[7] = evicted;
  free(U); free(where); free(miss); free(st);
  return ORC_OK;
}

/*
 * Union verification staging ("Memory split": verification staging;
 * "Speculative state": a verify block's queries fetch a missing row once).
 * The same resolution as orc_resolve, laid out so that each distinct row of
 * the verify block is staged once:
 *   loc[u]     u < U: location of the u-th distinct selected row, ascending
 *              row order; loc[u] = ORC_END_LOC for U <= u < Q*k;
 *   index[e]   position of sel[e] among those U rows.
 * U is counters[1].  On an error nothing changes, every loc is ORC_END_LOC
 * and every index -1.
 */
int orc_resolve_union(orc_pool *p, uint32_t step, int32_t r, int32_t s,
                      int32_t Q, int32_t k, const int32_t *sel, uint32_t *loc,
                      int32_t *index, uint32_t *counters) {
  if (Q < 0 || k < 0) return ORC_EINVAL;
  int64_t n = (int64_t)Q * k;
  uint32_t *per_entry = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)(n + 1));
  int32_t *U = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
  if (!per_entry || !U) {
    free(per_entry); free(U);
    return ORC_ENOMEM;
  }
  int rc = orc_resolve(p, step, r, s, Q, k, sel, per_entry, counters);
  for (int64_t e = 0; e < n; ++e) {
    loc[e] = ORC_END_LOC;
    index[e] = -1;
  }
  if (rc == ORC_OK) {
    memcpy(U, sel, sizeof(int32_t) * (size_t)n);
    qsort(U, (size_t)n, sizeof(int32_t), cmp_i32);
    int64_t nu = 0;
    for (int64_t e = 0; e < n; ++e)
      if (nu == 0 || U[nu - 1] != U[e]) U[nu++] = U[e];
    /* every entry of one row has the same location: take the entry's */
    for (int64_t e = 0; e < n; ++e) {
      int64_t u = find_sorted(U, nu, sel[e]);
      index[e] = (int32_t)u;
      loc[u] = per_entry[e];
    }
  }
  free(per_entry); free(U);
  return rc;
}

/* ------------------------------------------------------------ gather */

/*
 * staging[e] = the row bytes at loc[e] (zeros for ORC_NO_LOC; ORC_END_LOC
 * leaves staging[e] untouched).  Optional
 * slots hold copies of their owner's imported rows, which never change, so
 * they are read from the owner's host copy.  Every location must point at
 * a payload-tracked source, else ORC_EINVAL.
 */
int orc_gather(const orc_pool *p, const uint32_t *loc, int64_t n,
               uint16_t *staging) {
  if (!p || n < 0) return ORC_EINVAL;
  size_t E = (size_t)p->E;
  int64_t pairs = (int64_t)p->R * p->S;
  for (int64_t e = 0; e < n; ++e) {
    uint16_t *dst = staging + (size_t)e * E;
    uint32_t tier = loc[e] >> 30, idx = loc[e] & 0x3FFFFFFFu;
    const uint16_t *from = NULL;
    if (loc[e] == ORC_END_LOC) { /* past a union list: staging untouched */
      continue;
    } else if (loc[e] == ORC_NO_LOC) {
      memset(dst, 0, E * 2);
      continue;
    } else if (tier == ORC_TIER_TAIL) {
      int64_t pair = idx / p->T;
      if (pair >= pairs || !p->src[pair].tracked) return ORC_EINVAL;
      from = p->src[pair].tail + (size_t)(idx % p->T) * E;
    } else if (tier == ORC_TIER_OPT) {
      int64_t slot = idx / p->PR;
      if (slot >= p->capacity || p->slot_pair[slot] < 0) return ORC_EINVAL;
      const orc_source *o = &p->src[p->slot_pair[slot]];
      if (!o->tracked) return ORC_EINVAL;
      int64_t row = (int64_t)p->slot_page[slot] * p->PR + idx % p->PR;
      from = (o->imported ? o->imported : o->host) + (size_t)row * E;
    } else if (tier == ORC_TIER_HOT) {
      int64_t pair = idx / p->B;
      if (pair >= pairs || !p->src[pair].tracked) return ORC_EINVAL;
      from = p->src[pair].hot + (size_t)(idx % p->B) * E;
    } else {
      return ORC_EINVAL;
    }
    memcpy(dst, from, E * 2);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------ readers */

int orc_read_state(const orc_pool *p, int32_t r, int32_t s, int32_t *tags,
                   uint32_t *stamps, int32_t *page_slot, int64_t *lengths) {
  orc_source *src = get_src((orc_pool *)p, r, s);
  if (!src) return ORC_EINVAL;
  if (tags) memcpy(tags, src->tags, sizeof(int32_t) * (size_t)p->B);
  if (stamps) memcpy(stamps, src->stamps, sizeof(uint32_t) * (size_t)p->B);
  if (page_slot) memcpy(page_slot, src->page_slot, sizeof(int32_t) * (size_t)p->pages_max);
  if (lengths) { lengths[0] = src->N; lengths[1] = src->L; lengths[2] = src->admitted; }
  return ORC_OK;
}

/* which: 0 = host rows [row0, row0+n), 1 = tail ring slots, 2 = hot slots */
int orc_read_rows(const orc_pool *p, int32_t r, int32_t s, int which,
                  int64_t row0, int64_t n, uint16_t *out) {
  orc_source *src = get_src((orc_pool *)p, r, s);
  if (!src || !src->tracked || row0 < 0 || n < 0) return ORC_EINVAL;
  int64_t lim = which == 0 ? p->max_rows : which == 1 ? p->T : p->B;
  if (row0 + n > lim) return ORC_EINVAL;
  const uint16_t *base = which == 0 ? src->host : which == 1 ? src->tail : src->hot;
  if (!base) return ORC_EINVAL; /* a window source has no host copy */
  memcpy(out, base + (size_t)row0 * p->E, (size_t)n * p->E * 2);
  return ORC_OK;
}

/*
 * Invariants of one source: hot tags unique and inside [0, L); a filled
 * slot has a stamp >= 1 and an empty one stamp 0; ready optional pages are
 * complete imported pages owned by this pair in the slot table.  Returns 0
 * or the number of the first violated check.
 */
int orc_check(const orc_pool *p, int32_t r, int32_t s) {
  orc_source *src = get_src((orc_pool *)p, r, s);
  if (!src) return 100;
  int64_t pair = (int64_t)r * p->S + s;
  for (int32_t j = 0; j < p->B; ++j) {
    int32_t t = src->tags[j];
    if (t < -1 || (t >= 0 && t >= src->L)) return 1;
    if (t == -1 && src->stamps[j] != 0) return 2;
    if (t >= 0 && src->stamps[j] == 0) return 3;
    for (int32_t i = 0; i < j; ++i)
      if (t >= 0 && src->tags[i] == t) return 4;
  }
  for (int64_t q = 0; q < p->pages_max; ++q) {
    int32_t sl = src->page_slot[q];
    if (sl < 0) continue;
    if ((q + 1) * p->PR > src->N) return 5;
    if (sl >= p->capacity || p->slot_pair[sl] != pair || p->slot_page[sl] != q)
      return 6;
  }
  /* no row without a copy: each page is ready on the GPU or backed on the host */
  for (int64_t q = 0; q < p->pages_max; ++q) {
    if (src->page_slot[q] < 0 && !src->backed[q]) return 7;
    if (src->backed[q] && src->pend[q]) return 8;
    if (src->backed[q] && src->host && src->imported && (q + 1) * p->PR <= src->N &&
        memcmp(src->host + (size_t)q * p->PR * p->E, src->imported + (size_t)q * p->PR * p->E,
               (size_t)p->PR * p->E * 2) != 0)
      return 9;
  }
  return 0;
}
