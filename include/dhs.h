/*
 * dhs.h -- C ABI of the GB300 (sm_103a) hierarchical sparse KV resolve +
 * gather library (libdhs.so).
 *
 * The operation is the per-decode-step path of "Adaptive DHiSparse:
 * Speculative Decoding over a Load-Adaptive KV Hierarchy" (How it works):
 * each request's top-k selected KV rows are located, each at the first of
 * three places that holds it -- (1) the tail ring of recent rows or an
 * imported page resident on the GPU, (2) one of the B hot-cache slots, found
 * by their tags, least recently used slots making room, (3) otherwise its
 * pinned host copy, fetched into a victim hot-cache slot -- and the selected
 * rows are gathered into a contiguous staging buffer for sparse attention.
 *
 * Conventions for every call:
 *   - Return value: DHS_OK (0) or a negative DHS_E* code.  No call throws,
 *     aborts or prints.  A call that fails validation changes nothing.
 *   - Device work is asynchronous and ordered on the pool's stream; no call
 *     on the hot path (dhs_append, dhs_resolve, dhs_gather,
 *     dhs_resolve_gather) synchronises the host.
 *   - Errors found on the device (a selected row outside [0, L), more missing
 *     rows than unprotected hot slots, a gather location outside its arena)
 *     cannot be returned by the launching call: they leave the affected
 *     (request, source) unchanged for that step, zero its counters and set a
 *     sticky flag read by dhs_status().  Its entries that step 1 of
 *     "Resolution" resolves (the tail, or a ready page of the optional map:
 *     a lookup that changes no state) keep their locations; every other
 *     entry gets DHS_NO_LOC (a union item: an empty list, DHS_END_LOC and
 *     index -1).
 *   - A pool is not thread-safe: calls on one pool must not overlap.
 *   - Ownership: the caller owns every device buffer (the four arenas,
 *     selections, location vectors, staging, counters, appended rows) and
 *     every pinned host buffer; the library owns only host-side metadata.
 *
 * Location encoding: DHS_LOC(tier, index) = (tier << 30) | index, where
 *   tier DHS_TIER_TAIL: index = pair * tail_rows + row % tail_rows
 *   tier DHS_TIER_OPT : index = slot * page_rows + row % page_rows
 *   tier DHS_TIER_HOT : index = pair * hot_rows + hot slot
 * and pair = req * sources + src.  Row `index` of the tier's arena starts at
 * byte index * row_bytes.
 */
#ifndef DHS_H_
#define DHS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ error codes */
#define DHS_OK 0
#define DHS_EINVAL (-1)     /* bad argument, size, alignment or configuration */
#define DHS_ENOMEM (-2)     /* host metadata allocation failed */
#define DHS_EWOULDWAIT (-3) /* capacity cannot be covered: the admission waits */
#define DHS_EBUDGET (-4)    /* device: more missing rows than unprotected slots */
#define DHS_ERANGE (-5)     /* device: selected row or location out of range */
#define DHS_ETIMEDOUT (-6)  /* device: a bounded wait gave up (sticky flag) */
#define DHS_ECUDA (-7)      /* a CUDA runtime call or launch failed */
#define DHS_ESTATE (-8)     /* request/source not admitted, or already admitted */

/* ------------------------------------------------------------ locations */
#define DHS_TIER_TAIL 0u
#define DHS_TIER_OPT 1u
#define DHS_TIER_HOT 2u
#define DHS_NO_LOC 0xFFFFFFFFu
/* Past the end of a union location list (DHS_ITEM_UNION): gathers skip it. */
#define DHS_END_LOC 0xFFFFFFFEu
#define DHS_LOC(tier, index) ((((uint32_t)(tier)) << 30) | ((uint32_t)(index)))

/* Per-resolve counters (uint32 each), one block of DHS_NUM_COUNTERS per item:
 * entries = Q*k; unique = distinct selected rows over the verify block;
 * tail / opt = distinct rows found in step 1 (tail, optional map);
 * hot = distinct rows found by the hot-cache scan (step 2);
 * host = distinct rows copied from pinned host memory (step 3);
 * scan_max = probes of the longest hot-cache scan (slot + 1 on a hit, B on
 * a miss; never above B); evicted = victims that held a row. */
enum {
  DHS_CNT_ENTRIES = 0,
  DHS_CNT_UNIQUE,
  DHS_CNT_TAIL,
  DHS_CNT_OPT,
  DHS_CNT_HOT,
  DHS_CNT_HOST,
  DHS_CNT_SCAN_MAX,
  DHS_CNT_EVICTED,
  DHS_NUM_COUNTERS
};

/* Sticky device status flags (dhs_status). */
#define DHS_STATUS_ERANGE 1u  /* a selection held a row outside [0, L) */
#define DHS_STATUS_EBUDGET 2u /* a resolve needed more victims than slots */
#define DHS_STATUS_ELOC 4u    /* a gather location pointed outside its arena */
#define DHS_STATUS_ETIMEDOUT 8u /* a bounded device wait gave up; its tile was skipped */

/* ------------------------------------------------------------ pool */
typedef struct dhs_pool dhs_pool;

/*
 * Pool geometry ("Memory split": every request/KV-source pair owns B hot-cache
 * rows, its tail ring and its metadata, none of them lent out; whole pages of
 * imported history may occupy optional capacity that can be taken back).
 */
typedef struct {
  int32_t max_requests;          /* R: request slots 0..R-1 */
  int32_t sources;               /* S: KV sources per request (own state + payload) */
  int32_t row_bytes;             /* bytes per KV row: multiple of 16 (576 bf16 = 1152) */
  int32_t page_rows;             /* rows per optional page: power of two (64) */
  int32_t tail_rows;             /* T >= 1: the tail holds rows [L-T, L) */
  int32_t hot_rows;              /* B in [1, 16384]: hot-cache rows per (req, src) */
  int32_t max_queries;           /* Q: verify queries per resolve item */
  int32_t max_topk;              /* k: selected rows per query */
  int64_t max_rows_per_request;  /* bound on L = imported + appended rows */
  int64_t optional_pages;        /* optional capacity in pages */
  int64_t admission_reserve_pages; /* pages an admission must leave free */
  void *hot_dev;   /* [R][S][B] rows            (DHS_BUF_HOT bytes)  */
  void *tail_dev;  /* [R][S][T] rows            (DHS_BUF_TAIL bytes) */
  void *opt_dev;   /* [optional_pages][page_rows] rows (DHS_BUF_OPT bytes) */
  void *meta_dev;  /* tags, stamps, page maps, miss lists, status (DHS_BUF_META) */
  void *stream;    /* cudaStream_t for all device work (NULL = legacy default) */
} dhs_pool_config;

enum { DHS_BUF_HOT = 0, DHS_BUF_TAIL, DHS_BUF_OPT, DHS_BUF_META, DHS_NUM_BUFS };

/*
 * Bytes of the four device buffers the caller must allocate for `cfg`
 * (pointer and stream fields are ignored), written to out[DHS_NUM_BUFS].
 * Every buffer must be 256-byte aligned.  Pure host arithmetic.  The pages
 * have no passage for this call: it exists because the caller, not the
 * library, owns device memory (their "Memory split" fixes what the buffers
 * hold, not how they are sized).
 * Errors: DHS_EINVAL for an invalid geometry.
 */
int dhs_pool_bytes(const dhs_pool_config *cfg, size_t out[DHS_NUM_BUFS]);

/*
 * Create a pool on the calling thread's current CUDA device.  The library
 * keeps the pointers (it copies no payload) and enqueues on cfg->stream the
 * initialisation of meta_dev (empty hot caches: tag -1, stamp 0; no ready
 * pages).  Errors: DHS_EINVAL (geometry, null or misaligned buffer, or a
 * geometry whose resolve kernel would not fit in shared memory), DHS_ENOMEM,
 * DHS_ECUDA.
 */
int dhs_pool_create(const dhs_pool_config *cfg, dhs_pool **out);

/* Free the host metadata (device buffers stay the caller's).  NULL is a no-op.
 * Work already enqueued still runs; synchronise the stream before freeing
 * the buffers. */
void dhs_pool_destroy(dhs_pool *pool);

/*
 * Admit (req, src) with n_rows imported rows ("Resident-first admission").
 * host_rows: caller-owned pinned + mapped host memory (cudaHostAlloc or
 * cudaHostRegister with the mapped flag), 16-byte aligned, holding rows
 * [0, n_rows) and room
 * for max_rows_per_request rows (appended rows are written through to it);
 * it must outlive the admission.  resident_page_mask: one byte per complete
 * page (n_rows / page_rows of them), nonzero = keep on device; NULL = all
 * complete pages.  Resident pages take the lowest free optional slots, pages
 * ascending; their bytes are copied from host_rows before the next device
 * call observes them (pages reclaimed before then are never copied).  The
 * tail ring is filled with rows [max(0, n_rows-T), n_rows).
 * Capacity rule (Memory split): used + resident pages <= optional_pages -
 * admission_reserve_pages, else DHS_EWOULDWAIT with *deficit_pages set and
 * nothing changed; the caller may dhs_reclaim() and retry.
 * Errors: DHS_EINVAL, DHS_ESTATE (already admitted), DHS_EWOULDWAIT,
 * DHS_ECUDA.
 */
int dhs_admit(dhs_pool *pool, int32_t req, int32_t src, void *host_rows,
              int64_t n_rows, const uint8_t *resident_page_mask,
              int64_t *deficit_pages);

/*
 * "Reclamation and refill": walk `order` (n request ids) and take whole
 * requests' optional pages -- every source of the request -- until
 * deficit_pages are freed; other requests keep theirs.  If the listed
 * requests cannot cover the deficit nothing is taken and DHS_EWOULDWAIT is
 * returned.  Pages are freed in stream order, after every earlier reader on
 * the pool's stream; hot-cache rows stay valid (they are copies).
 * *freed_pages receives the pages taken.  Errors: DHS_EINVAL,
 * DHS_EWOULDWAIT.
 */
int dhs_reclaim(dhs_pool *pool, const int32_t *order, int32_t n,
                int64_t deficit_pages, int64_t *freed_pages);

/* Release every source of request `req`: free its pages, empty its hot
 * caches, forget its host rows.  Errors: DHS_EINVAL, DHS_ECUDA. */
int dhs_release(dhs_pool *pool, int32_t req);

/*
 * Resident-first admission of rows that are on the device ("Resident-first
 * admission": while HBM has room, an arriving request's imported history
 * stays on the GPU and its host backup is put off).  dev_rows: device memory, rows
 * [0, n_rows) of row_bytes each (e.g. the prefill's output), read only by
 * copies this call enqueues on the pool's stream (reuse it after the stream
 * has passed them).  host_rows: as for dhs_admit, but its imported rows need
 * not be written yet.  Pages are chosen and the capacity rule applied as in
 * dhs_admit.  This call enqueues: the tail ring fill and the resident pages'
 * copies from dev_rows (device to device), and the copy to host_rows of
 * every other imported row -- pages left out and the incomplete last page,
 * which only the host can serve (device to host).  The resident pages' own
 * host backup is deferred: they enter the backup order (admission order,
 * pages ascending), see dhs_backup; until then their host rows are not
 * valid.  Errors: as dhs_admit.
 */
int dhs_admit_device(dhs_pool *pool, int32_t req, int32_t src, const void *dev_rows,
                     void *host_rows, int64_t n_rows, const uint8_t *resident_page_mask,
                     int64_t *deficit_pages);

/*
 * Admit (req, src) as a window source ("Speculative state": a drafter
 * retains only the rows its window covers, stored as a ring).  The source's tail ring
 * of tail_rows rows is its only storage: it has no host copy, no optional
 * pages (it takes no pool capacity) and its rows never enter the hot cache.
 * A window of n_rows rows holds rows [n_rows - m, n_rows), m = min(n_rows,
 * tail_rows), at ring slots row mod tail_rows.
 *   dev_rows  device memory, 16-byte aligned: those m rows in order, row j
 *             at dev_rows + j * row_bytes; read only by copies this call
 *             enqueues on the pool's stream (reuse it after the stream has
 *             passed them).  May be NULL when n_rows is 0.
 * Afterwards: dhs_append writes a window source's rows into the ring only
 * (each overwrites the row tail_rows before it, which leaves the window for
 * good); a resolve gives every selected row in [L - tail_rows, L) its tail
 * location (counters: entries, unique, tail = unique, the rest 0), and a
 * selection holding any other row is DHS_ERANGE (device-side, as for rows
 * outside [0, L): the item keeps only its in-window locations).  Gathers,
 * release and the status calls treat it like any source.  The layout of the
 * location vector is unchanged (tier DHS_TIER_TAIL).
 * Errors: DHS_EINVAL (arguments, alignment, n_rows > max_rows_per_request),
 * DHS_ESTATE (already admitted), DHS_ECUDA.
 */
int dhs_admit_window(dhs_pool *pool, int32_t req, int32_t src, const void *dev_rows,
                     int64_t n_rows);

/*
 * Deferred host backup: enqueue the device-to-host copies of at most
 * max_pages pages in backup order; *done = pages backed up.  dhs_reclaim
 * backs up a reclaimed page that is still pending before freeing its slot
 * (Reclamation and refill: a page's slot is reused only once its host backup
 * is done and its earlier readers have finished): the copy is ordered on
 * the pool's stream after every earlier reader and before any later copy
 * into the slot.  Released requests' pages
 * need no backup.  Errors: DHS_EINVAL, DHS_ECUDA.
 */
int dhs_backup(dhs_pool *pool, int64_t max_pages, int64_t *done);

/* Pages whose host backup is still deferred. */
int64_t dhs_pending_backup(const dhs_pool *pool);

/*
 * Bounded round-robin refill ("Reclamation and refill": refill uses bounded
 * round-robin).  Requests are visited cyclically from a cursor that starts
 * at request 0; a visit to a request with a complete imported page that is
 * not optional-resident makes its lowest (source, page) such page resident
 * again in the lowest free slot, its bytes copied from the host copy (which
 * every non-resident page has) before the next device call observes it.
 * Stops after max_pages pages, when used reaches optional_pages -
 * admission_reserve_pages, or when a whole round of visits found nothing;
 * the cursor keeps the next request to visit.  *filled = pages refilled.
 * Errors: DHS_EINVAL.
 */
int dhs_refill(dhs_pool *pool, int64_t max_pages, int64_t *filled);

/* Optional pages in use (host metadata). */
int64_t dhs_pool_used(const dhs_pool *pool);

/*
 * Make every admitted page ready now ("Reclamation and refill": a page is
 * read only once its copy is complete): enqueue on the pool's stream the
 * page copies and page-map updates that admissions, reclaims and releases
 * left pending (dhs_append, dhs_resolve and dhs_gather otherwise do this
 * first).  Asynchronous.  Errors: DHS_EINVAL, DHS_ECUDA.
 */
int dhs_flush(dhs_pool *pool);

/* --------------------------------------------------------- decode step */

/* One append: `count` (<= tail_rows) decode rows for (req, src), row j at
 * rows_dev + j * row_bytes (device memory, caller-owned). */
typedef struct {
  int32_t req;
  int32_t src;
  int32_t count;
  int32_t reserved;
  const void *rows_dev;
} dhs_append_item;

/*
 * Append decode rows (Limits: decode rows are served the hot-cache way).
 * Row L+j of (req, src) goes to tail slot (L+j) mod T and is written through
 * to the pinned host copy, so every row that leaves the tail keeps a host
 * copy (Reclamation and refill: no row is without a copy on the GPU or on
 * the host).  L grows by count.  (req, src) pairs must be distinct.
 * Errors: DHS_EINVAL (count > T, L + count > max_rows_per_request, null
 * rows), DHS_ESTATE, DHS_ECUDA.
 */
int dhs_append(dhs_pool *pool, const dhs_append_item *items, int32_t n_items);

#define DHS_ITEM_GATHER_ONLY 1u /* skip resolution: gather loc_dev as given */
/* Union verification staging ("Memory split": verification staging;
 * "Speculative state": a verify block's queries fetch a missing row once):
 * each distinct row of the verify block is staged once.  Resolution writes
 *   loc_dev[u]   u < U: location of the u-th distinct selected row, in
 *                ascending row order; DHS_END_LOC for U <= u < Q*k;
 *   index_dev    int32 [Q][k]: position of sel[q][i] among the U rows;
 * U = counters[1] (distinct rows).  The gather then writes staging rows
 * [0, U) only and leaves the rest of staging_dev untouched; a Reuse item
 * (DHS_ITEM_GATHER_ONLY) given such a location vector does the same.  On
 * DHS_ERANGE / DHS_EBUDGET the list is empty: every loc_dev entry is
 * DHS_END_LOC and every index_dev entry -1.  Needs index_dev; pools whose
 * histories are too long for the union's shared-memory plan (about
 * 12 bytes per 64 rows more than a plain resolve) refuse it with DHS_EINVAL.
 * This layout is not the pages' own: they describe per-query staging and
 * shared retrieval, not how staging is laid out. */
#define DHS_ITEM_UNION 2u

/*
 * One item of a decode step: the Q x k selection of one layer of one
 * request.
 *   sel_dev      int32 [Q][k] device, selected row ids (duplicates allowed)
 *   loc_dev      uint32 [Q][k] device: written by resolution, read by gather
 *   staging_dev  [Q][k][row_bytes] device gather target (gather only)
 *   counters_dev uint32 [DHS_NUM_COUNTERS] device or NULL
 *   index_dev    int32 [Q][k] device (DHS_ITEM_UNION only, else ignored)
 * A DHS_ITEM_GATHER_ONLY item is a Reuse layer ("Model-specific reuse": a
 * Reuse layer takes over the location vector of the layer before it): it is
 * not resolved and
 * gathers loc_dev as given (req/src unused).
 */
typedef struct {
  int32_t req;
  int32_t src;
  int32_t queries;
  int32_t topk;
  uint32_t flags;
  int32_t reserved;
  const int32_t *sel_dev;
  uint32_t *loc_dev;
  void *staging_dev;
  uint32_t *counters_dev;
  int32_t *index_dev;
} dhs_item;

typedef struct {
  uint32_t step; /* >= 1; stamps record it; one verify block = one step */
  int32_t n_items;
  const dhs_item *items;
} dhs_step;

/*
 * "Resolution" for every item without DHS_ITEM_GATHER_ONLY.  Per item, over
 * the union of its Q verify queries ("Speculative state": the queries of a
 * verify block fetch each missing row once): each distinct row resolves in the
 * first place that holds it -- tail (rows >= L-T, checked first), the ready
 * optional map (complete imported pages), the hot cache (B tags; a hit
 * refreshes the slot's stamp to `step`) -- and the remaining rows, in
 * ascending row order, take the least recently used unprotected slots
 * (smallest (stamp, slot); slots hit or filled in this step are protected),
 * get their bytes copied from pinned host memory, and become hot.  Writes
 * loc_dev and counters_dev.  Items must name distinct (req, src) pairs.
 * Errors (synchronous): DHS_EINVAL, DHS_ESTATE, DHS_ECUDA; device-side
 * DHS_ERANGE / DHS_EBUDGET go to dhs_status() (the item keeps only its
 * step-1 locations, see above).
 */
int dhs_resolve(dhs_pool *pool, const dhs_step *step);

/*
 * dhs_resolve on a caller's side stream ("Model-specific reuse": layers that
 * share sparse indices but keep distinct payloads have their positions
 * prefetched).  The resolve and host-copy kernels are enqueued on
 * side_stream (a cudaStream_t of the pool's device) after everything the
 * pool's stream holds so far; the pool's stream waits for them before its
 * next device work (the next dhs_gather, for instance), while work the
 * caller enqueues on its own streams in between -- the previous layer's
 * compute -- overlaps them.  Results are those of dhs_resolve.  Errors: as
 * dhs_resolve, plus DHS_EINVAL for a null side_stream.
 */
int dhs_prefetch(dhs_pool *pool, const dhs_step *step, void *side_stream);

/*
 * Gather ("Memory split": verification staging holds the selected rows that
 * sparse attention reads; "Speculative state": each verify query's rows are
 * staged; "Model-specific reuse": Reuse layers gather an inherited location
 * vector).  staging_dev[q][i] = the row at loc_dev[q][i] for every item
 * (resolved or gather-only); DHS_NO_LOC rows become zeros and DHS_END_LOC
 * entries are skipped (staging untouched).  staging_dev must
 * be 16-byte aligned.  Stream-ordered after any earlier dhs_resolve.
 * Errors: DHS_EINVAL, DHS_ECUDA; out-of-arena locations -> zeros +
 * DHS_STATUS_ELOC.
 */
int dhs_gather(dhs_pool *pool, const dhs_step *step);

/*
 * dhs_resolve for callers that cannot allocate device memory where they
 * resolve (an embedding runtime that hands the library only the buffers it
 * owns, or code running where allocation calls are not permitted).  The
 * results are the same as dhs_resolve's; the only difference is where the
 * per-item miss lists (rows to fetch from host memory and their hot slots)
 * live: in one fixed 540,672-byte device array inside libdhs.so instead of the
 * pool's metadata buffer.  The call allocates nothing (no cudaMalloc,
 * cudaFree or allocating library routine).  The pages describe no such
 * entry point; it has no counterpart there.
 *   - Limit: the pool's R*S*min(B, max_queries*max_topk) must be at most
 *     65536 and R*S at most 4096; larger pools get DHS_EINVAL and nothing
 *     is launched.
 *   - The array is shared by every call in the process and keeps the last
 *     call's contents; every entry a call reads is written earlier in the
 *     same call, so nothing needs clearing.  Calls that overlap on the GPU
 *     (other streams, other pools) race on it: issue them in one stream
 *     order.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     A cudaDeviceReset unloads the array with the library's device code,
 *     so the kept address is stale afterwards: do not use this entry point
 *     on a device after resetting it.
 *   - An outstanding dhs_prefetch is waited for only when the step names
 *     one of its (request, source) pairs, as in dhs_resolve.
 * Errors: as dhs_resolve, plus DHS_EINVAL for pools beyond the limit.
 */
int dhs_resolve_noalloc(dhs_pool *pool, const dhs_step *step);

/*
 * dhs_gather enqueued on a caller's stream (a cudaStream_t of the pool's
 * device) instead of the pool's: it runs after everything the pool's stream
 * holds so far, and the pool's next call that can change rows (resolve,
 * append, admission, reclaim, release, ...) waits for it.  With two staging
 * buffers this lets a layer's gather overlap the previous layer's compute;
 * the caller orders its own consumers after the gather on `stream`.
 * Results are those of dhs_gather.  Errors: as dhs_gather, plus DHS_EINVAL
 * for a null stream.
 */
int dhs_gather_on(dhs_pool *pool, const dhs_step *step, void *stream);

/*
 * dhs_resolve followed by dhs_gather on the same step, with the same results.
 * The kernels overlap (programmatic dependent launch): rows that resolve in
 * step 1 (tail, ready optional page) are copied into staging while the
 * resolve kernel still runs; rows that need the hot cache wait for it.
 */
int dhs_resolve_gather(dhs_pool *pool, const dhs_step *step);

/*
 * One whole decode step: dhs_append(appends) then dhs_resolve_gather(step),
 * with the same results.  When every appending pair is also resolved in
 * `step`, the appends are carried out by the resolve kernel itself (one
 * launch fewer), and the gather copies those new rows only after the resolve
 * kernel has finished.  Otherwise it runs the three calls in order.
 * Errors: as dhs_append and dhs_resolve_gather; on a validation error
 * nothing is appended or launched.
 */
int dhs_decode_step(dhs_pool *pool, const dhs_append_item *appends, int32_t n_appends,
                    const dhs_step *step);

/* One contiguous copy between host and device memory (see
 * dhs_decode_step_host).  Host memory should be pinned for the copies to be
 * asynchronous. */
typedef struct {
  void *dst;
  const void *src;
  size_t bytes;
} dhs_copy;

/*
 * dhs_decode_step with its inputs and outputs in host memory: enqueue the
 * n_in host-to-device copies (the step's selections and decode rows, into
 * the device buffers its items and appends name), the decode step, the
 * n_out device-to-host copies (locations, counters), then synchronise the
 * pool's stream; on return the outputs are in host memory.  One
 * cudaMemcpyAsync per copy on the pool's stream.  Errors: as
 * dhs_decode_step, DHS_EINVAL for a copy with a null pointer, DHS_ECUDA.
 */
int dhs_decode_step_host(dhs_pool *pool, const dhs_copy *in, int32_t n_in,
                         const dhs_append_item *appends, int32_t n_appends,
                         const dhs_step *step, const dhs_copy *out, int32_t n_out);

/*
 * dhs_decode_step_host without the final synchronisation, for a pipelined
 * caller: it returns once everything is enqueued.
 *   - The n_in host-to-device copies go on `in_stream` (a cudaStream_t; NULL
 *     = the pool's stream) with no other ordering: the caller makes that
 *     stream wait until earlier work is done with the input buffers.  The
 *     step waits for them.
 *   - The step runs on the pool's stream, after everything already on it.
 *   - The n_out device-to-host copies go on `out_stream` (NULL = the pool's
 *     stream) after the step.  The caller waits for them (an event it records
 *     on that stream) before it reads the outputs, and makes the pool's
 *     stream wait for them before a later step writes the same device
 *     buffers: the pool does not track readers of the caller's buffers.
 * With separate streams and alternating buffers, step s+1's inputs come in
 * and step s-1's outputs go out while step s runs.  Errors: as
 * dhs_decode_step_host (device-side errors go to dhs_status).
 */
int dhs_decode_step_host_async(dhs_pool *pool, const dhs_copy *in, int32_t n_in,
                               void *in_stream, const dhs_append_item *appends,
                               int32_t n_appends, const dhs_step *step,
                               const dhs_copy *out, int32_t n_out, void *out_stream);

/*
 * Synchronise the pool's stream, read and clear the sticky device status.
 * The pages have no passage for this call: device-side errors cannot be
 * returned by the asynchronous call that caused them, so they are read here.
 * *flags (may be NULL) receives DHS_STATUS_* bits.  Returns DHS_OK when no
 * flag was set, else DHS_ERANGE (ERANGE or ELOC), DHS_EBUDGET or
 * DHS_ETIMEDOUT, or DHS_ECUDA if the stream reported an error.
 */
int dhs_status(dhs_pool *pool, uint32_t *flags);

/*
 * Read one source's hot-cache state and page map (synchronises the stream;
 * for tests and diagnostics).  tags int32[B], stamps uint32[B],
 * page_slot int32[ceil(max_rows_per_request / page_rows)] (host view, -1 =
 * not ready), info int64[4] = {imported rows N, length L, admitted, last
 * resolve status (0, DHS_ERANGE or DHS_EBUDGET)}.  Any pointer may be NULL.
 */
int dhs_read_state(dhs_pool *pool, int32_t req, int32_t src, int32_t *tags,
                   uint32_t *stamps, int32_t *page_slot, int64_t *info);

/* Tunables (performance only; results do not depend on them). */
/* Host-copy CTAs; 0 = automatic.  The pages size the copy kernel's grid
 * between 4 and 32 blocks by batch size; on GB300 fewer than about 16 blocks
 * leave the host link idle (miss-heavy workload: 4 blocks 78 GB/s, 16 188,
 * 32 198 of a 211 GB/s pinned copy), so the automatic grid is never below
 * 32.  It grows past 32 until each block's items span at most 1 GiB of
 * pinned rows (max_rows_per_request * row_bytes per item), up to one block
 * per item and per SM: a block whose rows lie in a larger region re-walks
 * address translations and copies at a fraction of the link's rate.  A
 * launch of more items than SMs whose copy blocks claim rows
 * (DHS_OPT_COPY_STEAL) runs 64 blocks of 256 threads instead of 32 of 512.
 * A value set here keeps 512 threads a block. */
#define DHS_OPT_COPY_CTAS 1
#define DHS_OPT_GATHER_IMPL 2 /* 1 = TMA bulk copy, 16-row tiles of two
                                     warps (default); 0 = 16-byte vector copy,
                                     256 threads per 32-row tile (the only one
                                     for rows too large to stage 16 of them) */
/* Timeline: value = address of a device buffer of 8 uint64 (0 = off).  Each
 * kernel kind k (0 resolve, 1 host copy, 2 gather, 3 fresh-row copy) atomically
 * lowers buf[2k]
 * to its earliest CTA start and raises buf[2k+1] to its latest CTA end
 * (%globaltimer, ns; the host copy's start is when its copying begins, after
 * it has waited for the resolve kernel); the caller initialises buf[2k] to
 * UINT64_MAX and buf[2k+1] to 0. */
#define DHS_OPT_TRACE 3
/* 1 (default): fused gathers copy step-1 rows while the resolve kernel runs,
 * and every other row as soon as the resolve kernel has written its item's
 * locations, except rows in hot slots this step's host copy fills; 0: they
 * wait for the resolve and host-copy kernels first. */
#define DHS_OPT_EARLY 4
/* Fused steps (TMA gather): rows in hot slots that this step's host copy
 * fills go to a device list copied by one more kernel after the copy, so
 * gather tiles never wait for the copy.  -1 (default) = on when more than a
 * tenth of the admitted complete pages are not optional-resident; 0 = off
 * (such rows wait in their tile); 1 = on. */
#define DHS_OPT_FRESH_LIST 5
/* TMA gather: consecutive 16-entry tiles per CTA, 1 (default) .. 64. */
#define DHS_OPT_GATHER_TPC 6
/* Fused steps (TMA gather, early copies on): 1 (default) = the host copy
 * writes each row it fetches into the hot cache and into every staging
 * entry of the resolved item that selected it, and the gather leaves those
 * rows out; 0 = the gather copies them from the hot cache after the copy. */
#define DHS_OPT_STAGE_MISSES 7
/* Fused steps: how many times a gather tile polls for its item's published
 * locations, and a host-copy block for an item's published miss list,
 * before it gives up and waits for the whole resolve (and host-copy) grids
 * instead -- the slower path, with the same results.  -1 (default) = 2^20
 * polls; 0 .. 2^20.  0 sends every such tile and block down that path at
 * once (for tests of it). */
#define DHS_OPT_MARK_POLLS 8
/* The host copy starts while the resolve kernel runs (programmatic dependent
 * launch: 1) or after it (0).  -1 (default) = 1 while a launch's items span
 * at most 16 GiB of pinned rows, or when the launch's items plus its copy
 * blocks number at most the GPU's SMs (every copy block then finds an SM the
 * resolve grid leaves free); else 0.  Past 16 GiB the copy's blocks must land
 * on the same SMs step after step for the GPU to keep their address
 * translations, which a launch onto an idle GPU, or onto SMs left free, gives. */
#define DHS_OPT_COPY_PDL 9
/* Resolve launches of more than 32 items: -1 (default) = 512-thread CTAs two
 * per SM (one wave for more items than SMs) when the host copy launches after
 * the resolve grid and two CTAs' shared memory fits an SM, else 1024-thread
 * CTAs one per SM; 0 = always the latter; 1 = the former whenever it fits. */
#define DHS_OPT_RESOLVE_PAIRED 10
/* How the host copy's blocks share a launch's miss rows.  1: every item's
 * rows are claimed four at a time through a per-item cursor, and a block
 * whose own items are done claims the rows left in the others; 0: each block
 * copies its own items' rows.  -1 (default) = 1 while a launch's items span at
 * most 16 GiB of pinned rows, else 0 (past that a block reading another
 * item's rows walks translations its SM does not hold). */
#define DHS_OPT_COPY_STEAL 11
/* Resolve grid: 0 (default) = automatic (one CTA per item, except that a
 * launch of more items than SMs whose host copy overlaps the resolve kernel
 * runs one CTA for each SM the copy's blocks leave free, each resolving
 * several items in turn); n > 0 = at most n CTAs, each resolving items b,
 * b + n, ... */
#define DHS_OPT_RESOLVE_CTAS 12
int dhs_set_option(dhs_pool *pool, int32_t key, int64_t value);
/* The value in effect (DHS_OPT_FRESH_LIST: 0 or 1, the auto rule resolved
 * for the pool's current admissions).  DHS_EINVAL for an unknown key. */
int dhs_get_option(dhs_pool *pool, int32_t key, int64_t *value);

/* Static string for a DHS_* code. */
const char *dhs_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* DHS_H_ */
