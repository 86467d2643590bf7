// Host-side pool manager and C ABI of libdhs (see include/dhs.h).
//
// "Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
// Hierarchy", How it works:
//   Memory split -- every (request, KV source) pair owns B hot-cache rows,
//     its tail ring and its metadata, none of which is lent out; whole pages
//     of imported history may occupy optional capacity that can be taken
//     back, as long as required, optional and the admission reserve
//     together fit the pool.  Required memory is laid out per request slot
//     up front, so the rule is checked on the optional arena.
//   Resident-first admission -- resident pages take optional slots at
//     admission (lowest free slot first, pages ascending).
//   Reclamation and refill -- whole requests' pages are taken in reclaim
//     order until the deficit is covered, otherwise the admission waits.
//     Every device read of a page is ordered on the pool's stream, so a page
//     freed here is reused only by work enqueued after every earlier reader.
//
// Host metadata only: the caller owns every device buffer and every pinned
// host buffer.  Page bytes of an admission are copied lazily, just before
// the next device call that could observe them, so pages reclaimed before
// any step (e.g. an admission storm under memory pressure) are never moved.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <new>
#include <set>
#include <vector>

#include "dhs.h"
#include "dhs_internal.h"

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct MetaLayout {
  size_t tags, stamps, map, miss_rows, miss_slots, miss_count, copy_cursor, pair_status;
  size_t loc_ready, copy_ready, fill, later_count, status, later, miss_off, miss_ent;
  size_t total;
};

inline int64_t pages_max_of(const dhs_pool_config& c) {
  return (c.max_rows_per_request + c.page_rows - 1) / c.page_rows;
}

inline int64_t fill_words_of(const dhs_pool_config& c) { return (c.hot_rows + 31) / 32; }

// Fresh-row list entries: one resolved step's entries (Reuse layers beyond
// that copy their fresh rows in their own tiles).
inline int64_t later_cap_of(const dhs_pool_config& c) {
  return std::max<int64_t>(1, (int64_t)c.max_requests * c.sources * c.max_queries * c.max_topk);
}

// Staging entries one resolve of a (request, source) can list.
inline int64_t ent_cap_of(const dhs_pool_config& c) {
  return std::max<int64_t>(1, (int64_t)c.max_queries * c.max_topk);
}

inline int64_t mcap_of(const dhs_pool_config& c) {
  int64_t qk = (int64_t)c.max_queries * c.max_topk;
  return std::max<int64_t>(1, std::min<int64_t>(c.hot_rows, qk));
}

MetaLayout meta_layout(const dhs_pool_config& c) {
  MetaLayout m{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const size_t pairs = (size_t)c.max_requests * c.sources;
  m.tags = take(pairs * c.hot_rows * 4);
  m.stamps = take(pairs * c.hot_rows * 4);
  m.map = take(pairs * (size_t)pages_max_of(c) * 4);
  m.miss_rows = take(pairs * (size_t)mcap_of(c) * 4);
  m.miss_slots = take(pairs * (size_t)mcap_of(c) * 4);
  m.miss_count = take(pairs * 4);
  m.copy_cursor = take(pairs * 4);
  m.pair_status = take(pairs * 4);
  m.loc_ready = take(pairs * 4);
  m.copy_ready = take(pairs * 4);
  m.fill = take(pairs * (size_t)fill_words_of(c) * 4);
  m.later_count = take(2 * 4);
  m.status = take(64);
  m.later = take((size_t)later_cap_of(c) * sizeof(dhs::LaterEntry));
  m.miss_off = take(pairs * (size_t)(mcap_of(c) + 1) * 4);
  m.miss_ent = take(pairs * (size_t)ent_cap_of(c) * 4);
  m.total = off;
  return m;
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

int log2i(int64_t x) {
  int r = 0;
  while ((int64_t(1) << r) < x) ++r;
  return r;
}

// Shared-memory plan of the resolve kernel at the pool's largest sizes.
size_t max_resolve_smem(const dhs_pool_config& c, bool uni) {
  const int64_t w64 = (c.max_rows_per_request + 63) / 64;
  const int64_t qk = std::min<int64_t>(
      std::min<int64_t>((int64_t)c.max_queries * c.max_topk, c.max_rows_per_request),
      c.hot_rows);
  return dhs::resolve_smem_bytes((int)w64, (int)qk, c.hot_rows, uni, 0);
}

int validate_geometry(const dhs_pool_config* c) {
  if (!c) return DHS_EINVAL;
  if (c->max_requests <= 0 || c->sources <= 0 || c->tail_rows <= 0) return DHS_EINVAL;
  if (c->hot_rows <= 0 || c->hot_rows > dhs::kMaxHotRows) return DHS_EINVAL;
  if (c->row_bytes < 16 || c->row_bytes % 16 != 0 || c->row_bytes > 65536) return DHS_EINVAL;
  if (!is_pow2(c->page_rows) || c->page_rows > 65536) return DHS_EINVAL;
  if (c->max_queries < 0 || c->max_topk < 0) return DHS_EINVAL;
  if ((int64_t)c->max_queries * c->max_topk > (int64_t)1 << 20) return DHS_EINVAL;
  if (c->max_rows_per_request <= 0 || c->max_rows_per_request > INT32_MAX) return DHS_EINVAL;
  if (c->optional_pages < 0 || c->admission_reserve_pages < 0 ||
      c->admission_reserve_pages > c->optional_pages)
    return DHS_EINVAL;
  const int64_t pairs = (int64_t)c->max_requests * c->sources;
  const int64_t lim = (int64_t)1 << 30;  // location index bits
  if (pairs * c->tail_rows >= lim || pairs * c->hot_rows >= lim ||
      c->optional_pages * c->page_rows >= lim || pairs >= (1 << 24))
    return DHS_EINVAL;
  return DHS_OK;
}

struct PairState {
  bool admitted = false;
  bool window = false;          // window source: the tail ring is its only storage
  int64_t N = 0, L = 0;
  uint8_t* host = nullptr;      // caller's pinned host rows
  uint8_t* host_dev = nullptr;  // device-visible address of the same rows
  std::vector<int32_t> pending;  // resident pages whose bytes are not yet copied
  std::vector<uint64_t> backup;  // per page: backup order while the host copy is
                                 // deferred, 0 = backed (empty: all backed)
};

}  // namespace

struct dhs_pool {
  dhs_pool_config cfg{};
  cudaStream_t stream = nullptr;
  int device = 0;
  int64_t pairs = 0, pmax = 0, mcap = 0;
  int page_shift = 0;
  MetaLayout layout{};
  int32_t* tags = nullptr;
  uint32_t* stamps = nullptr;
  int32_t* map = nullptr;
  int32_t* miss_rows = nullptr;
  int32_t* miss_slots = nullptr;
  uint32_t* miss_count = nullptr;
  uint32_t* copy_cursor = nullptr;
  int32_t* pair_status = nullptr;
  uint32_t* status = nullptr;
  std::vector<PairState> ps;
  std::vector<int32_t> map_host;  // [pairs][pmax] mirror of the device map
  std::vector<int32_t> slot_pair, slot_page;
  int64_t first_free = 0, used = 0;
  int64_t dirty_lo = INT64_MAX, dirty_hi = -1;  // pairs whose map changed
  bool any_pending = false;
  int copy_ctas = 0;
  bool union_ok = false;  // the union staging plan fits in shared memory
  int gather_impl = dhs::kGatherTma;
  bool tma_ok = true;  // the TMA gather's tile fits the row size
  int gather_tpc = 1;   // DHS_OPT_GATHER_TPC
  int early = 1;        // fused gathers copy step-1 rows before the resolve ends
  uint32_t seq = 0;             // resolve launches so far
  uint32_t* loc_ready = nullptr;  // [pairs] per-item "locations written" marks
  uint32_t* copy_ready = nullptr; // [pairs] per-item "miss lists written" marks
  uint32_t* fill = nullptr;       // [pairs][fill_words] slots the step's copy fills
  uint32_t* later_count = nullptr;
  dhs::LaterEntry* later = nullptr;
  int64_t later_cap = 0;
  int fill_words = 0;
  uint32_t gen = 0;             // fused steps that launched a resolve
  bool fused_resolved = false;  // the current fused step launched one
  int fresh_list = -1;          // DHS_OPT_FRESH_LIST: -1 auto, 0 off, 1 on
  int64_t complete_pages = 0;   // complete imported pages of admitted pairs
  uint64_t bseq = 0;            // pages put in backup order so far
  std::set<std::pair<uint64_t, int64_t>> backup_order;  // (order, pair * pmax + page)
  int32_t rr = 0;               // refill cursor: the next request visited
  int sm_count = 0;
  int smem_optin = 0;           // opt-in shared memory per block
  int32_t* miss_off = nullptr;  // [pairs][Mcap + 1] staging entries of each miss
  int32_t* miss_ent = nullptr;  // [pairs][ent_cap]
  int64_t ent_cap = 0;
  int stage_misses = 1;         // DHS_OPT_STAGE_MISSES
  uint32_t mark_polls = dhs::kMarkPolls;  // DHS_OPT_MARK_POLLS
  int copy_pdl = -1;            // DHS_OPT_COPY_PDL: -1 auto, 0 off, 1 on
  int resolve_paired = -1;      // DHS_OPT_RESOLVE_PAIRED: -1 auto, 0 off, 1 whenever it fits
  int copy_steal = -1;          // DHS_OPT_COPY_STEAL: -1 auto, 0 off, 1 on
  int resolve_ctas = 0;         // DHS_OPT_RESOLVE_CTAS: 0 auto, > 0 at most that many
  int smem_per_sm = 0;          // shared memory per SM
  std::vector<uint8_t> staged_pair;  // the host copy stages this pair's misses this step
  std::vector<uint8_t> staged_item;  // per item of the step: a gather-only item whose
                                     // staging the host copy writes too
  unsigned long long* trace = nullptr;  // DHS_OPT_TRACE buffer, null = off
  // reusable launch tables
  std::vector<dhs::ResolveItem> ritems;
  std::vector<dhs::CopyItem> citems;
  std::vector<dhs::GatherItem> gitems;
  // gathers of a fused step: the resolved items' location vectors, sorted,
  // to find which pair (if any) published a gather item's locations
  struct LocKey {
    const void* loc;
    int32_t order;  // item index: of equal vectors the last one counts
    int64_t pair;
    bool operator<(const LocKey& o) const {
      return loc != o.loc ? std::less<const void*>()(loc, o.loc) : order < o.order;
    }
  };
  std::vector<LocKey> loc_keys;
  std::vector<dhs::AppendItem> aitems;
  std::vector<uint8_t> seen;
  std::vector<int32_t> app_of_pair;  // decode step: append item of each pair, -1 = none
  std::vector<int64_t> l0_of_pair;   // length of each resolved pair before this step's append
  std::vector<const uint8_t*> app_of_pair_rows;  // its appended rows' source, or null
  std::vector<uint32_t> seq_of_pair; // resolve launch that last resolved each pair
  std::vector<dhs::PageMove> moves;  // page list of the next page-move launch
  // dhs_prefetch: resolves enqueued on a caller's side stream; the pool's
  // stream waits for them before its next device work
  cudaEvent_t ev_main = nullptr, ev_prefetch = nullptr;
  // dhs_decode_step_host_async on callers' copy streams: the step waits for
  // the inputs (ev_in), the outputs' copies wait for the step (ev_step)
  cudaEvent_t ev_in = nullptr, ev_step = nullptr;
  bool prefetch_pending = false;
  bool join_gathers = true;  // enter(): also join gathers on other streams
  std::vector<uint8_t> pf_pair;  // pairs resolved by the outstanding prefetch
  // dhs_gather_on: gathers on callers' streams read rows the pool's next
  // resolve / append / admission may change; one event per such call,
  // joined (and recycled) by the pool's next call that can change rows
  std::vector<cudaEvent_t> ev_free, ev_gathers;
  ~dhs_pool() {
    if (ev_main) cudaEventDestroy(ev_main);
    if (ev_prefetch) cudaEventDestroy(ev_prefetch);
    if (ev_in) cudaEventDestroy(ev_in);
    if (ev_step) cudaEventDestroy(ev_step);
    for (cudaEvent_t e : ev_free) cudaEventDestroy(e);
    for (cudaEvent_t e : ev_gathers) cudaEventDestroy(e);
  }
};

namespace {

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? DHS_OK : DHS_ECUDA; }

// Host-copy launch policy.
//
// Grid: at least the upper end of the pages' 4-to-32-block scaling.  On
// GB300 the host link needs about 1024 rows in flight (16 blocks x 16 warps x
// 4 rows); below that the copy is latency-bound (miss-heavy workload: 4
// blocks 78 GB/s, 8 130, 16 188, 32 198 of the 211 GB/s pinned peak), and in
// same-box runs 32 blocks were as fast as or faster than 16 on every
// workload with misses, so the grid never shrinks below 32.
//
// Address translation of the pinned rows: a block copies the items b, b + G,
// ... of a launch, so its host footprint is the sum of those items' pinned
// regions.  Measured with the copy alone on GB300: while a block's footprint
// stays within about 1 GiB and each block lands on the same SM step after
// step, the copy runs at the link's rate even over a 58 GB pinned region
// (wide workload, 64 items of 0.9 GB: 64 blocks 199 GB/s); at 1.8 GiB per
// block it falls to 40-52 GB/s (32 blocks).  So the grid grows until every
// block's share of the items fits 1 GiB, up to one block per item and one per
// SM.
bool copy_steal(const dhs_pool* p, int64_t n_items);
bool copy_halves(const dhs_pool* p, int64_t n_items);
int copy_ctas(const dhs_pool* p, int64_t n_items) {
  if (p->copy_ctas > 0) return p->copy_ctas;
  if (copy_halves(p, n_items)) return std::min(64, std::max(1, p->sm_count));
  const int64_t item_span = p->cfg.max_rows_per_request * (int64_t)p->cfg.row_bytes;
  const int64_t per_block = std::max<int64_t>(1, (int64_t(1) << 30) / std::max<int64_t>(1, item_span));
  const int64_t want = (n_items + per_block - 1) / per_block;
  const int64_t cap = std::max<int64_t>(1, std::min<int64_t>(n_items, std::max(1, p->sm_count)));
  return (int)std::max<int64_t>(32, std::min(want, cap));
}

// Resolve launches of more items than SMs would take two waves of 1024-thread
// CTAs, one per SM.  When the host copy waits for the whole resolve grid
// anyway (copy_pdl false) and two CTAs' shared-memory plans fit one SM,
// 512-thread CTAs two per SM resolve every item in one wave instead, and the
// copy and the gather behind it start that much earlier.  With the copy
// overlapped (C64) the grid is instead one 1024-thread CTA per SM the copy
// leaves free (resolve_ctas): two CTAs per SM would spread over every SM and
// leave the copy's blocks none.
bool copy_pdl(const dhs_pool* p, int64_t n_items);
bool resolve_paired(const dhs_pool* p, int64_t n_items, size_t plan) {
  if (p->resolve_paired == 0 || n_items <= dhs::kResolveItemsSmall) return false;
  const bool fits = 2 * (plan + 1024) <= (size_t)p->smem_per_sm;
  if (p->resolve_paired == 1) return fits;
  return fits && n_items > p->sm_count && !copy_pdl(p, n_items);
}

// Programmatic dependent launch of the host copy (its blocks start while the
// resolve grid still runs and copy each item once its miss list is out) pays
// while the launch's pinned regions are small enough for the GPU's
// translation caches to hold them whatever SMs the blocks land on (C64: 9.7
// GB, 205 GB/s).  Past that it still pays when every copy block finds an SM
// that the resolve grid leaves free (a 1024-thread resolve CTA and a
// flat-list copy block each hold a whole SM's registers, so they never share
// an SM): the blocks are then all placed at launch, on the same SMs every
// step.  Otherwise blocks
// placed on whichever SMs the resolve grid frees land on different SMs from
// step to step and re-walk their translations, so the copy launches after
// the resolve grid, onto an idle GPU, where block b lands on the same SM
// every step (copy alone, pinned span 57 GB, 96 items and 96 blocks: 44-53 GB/s
// with the early start, 149 without it; 30 GB, 256 items and 32 blocks:
// 58-84 against 182).  One layer of the same 57 GB pool, 32 items beside 32
// blocks, runs faster overlapped, and much faster when other streams keep
// the GPU busy, since no launch then finds it idle (per-layer decode with
// side-stream prefetch and gathers on a second stream: 0.97-1.07 ms a step
// against 2.02-2.16).
bool copy_pdl(const dhs_pool* p, int64_t n_items) {
  if (p->copy_pdl >= 0) return p->copy_pdl == 1;
  const int64_t item_span = p->cfg.max_rows_per_request * (int64_t)p->cfg.row_bytes;
  if (n_items * item_span <= (int64_t(16) << 30)) return true;
  return n_items + copy_ctas(p, n_items) <= (int64_t)p->sm_count;
}

// Claiming rows through per-item cursors (and blocks done with their own
// items taking the rest of others') evens out the copy blocks' finishing
// times while the launch's pinned regions stay within the GPU's translation
// reach (C64, alternated on one box: 1738 us a step against 1762-1766).
// Past that a block that takes another item's rows reads from a region whose
// translations its SM does not hold, and the claims themselves cost an
// atomic round trip per item and warp where items have few misses each
// (C128: about 57 rows an item; its copy span 120 us against 94), so each
// block keeps to its own items there.
bool copy_steal(const dhs_pool* p, int64_t n_items) {
  if (p->copy_steal >= 0) return p->copy_steal == 1;
  const int64_t item_span = p->cfg.max_rows_per_request * (int64_t)p->cfg.row_bytes;
  return n_items * item_span <= (int64_t(16) << 30);
}

// Resolve grid.  A launch of more items than SMs whose host copy overlaps it
// (within the translation reach) runs one CTA per SM it leaves to the copy:
// sm_count - copy blocks CTAs resolve every item, a few each in turn, all of
// them resident from the start.  The copy grid, a programmatic dependant,
// launches only once every resolve CTA has started, so with one CTA per
// item its blocks waited for the second wave's CTAs to be placed and took
// their SMs only then (C64: copying began 52 us into the step); now they
// are placed at once and start on each item as its miss list comes out.
int resolve_ctas(const dhs_pool* p, int64_t n_items, bool paired) {
  if (p->resolve_ctas > 0) return (int)std::min<int64_t>(n_items, p->resolve_ctas);
  if (paired || n_items <= p->sm_count || !copy_pdl(p, n_items)) return (int)n_items;
  return std::max(1, p->sm_count - copy_ctas(p, n_items));
}

// Block size.  A claiming launch of more items than SMs (C64: 256 items,
// its resolve grid one CTA per SM the copy leaves free) runs the copy as 64
// blocks of 256 threads instead of 32 of 512: as many rows in flight, over
// twice the SMs, each with room left for gather CTAs beside its block
// (C64, alternated on one box: 1715-1716 us median against 1723-1724).
// Smaller launches keep 32 blocks of 512: C8 and the miss-heavy workload
// were slower with the halved blocks (24.82-24.85 us against 24.66-24.68,
// 137 against 133).
bool copy_halves(const dhs_pool* p, int64_t n_items) {
  return p->copy_ctas <= 0 && n_items > p->sm_count && copy_steal(p, n_items);
}
int copy_threads(const dhs_pool* p, int64_t n_items) {
  return copy_halves(p, n_items) ? dhs::kCopyThreads / 2 : dhs::kCopyThreads;
}

// Where each block keeps to its own items (past the translation reach), it
// also keeps its SM to itself: it reserves all but 2 KB of the shared memory
// a block may take, so no gather CTA lands beside it and evicts its host
// rows' translations from the SM's caches with its own device addresses.
size_t copy_hold_limit(int smem_optin) { return (size_t)std::max(0, smem_optin - 2048); }
size_t copy_hold_smem(const dhs_pool* p, int64_t n_items) {
  return copy_steal(p, n_items) ? 0 : copy_hold_limit(p->smem_optin);
}

// Pages small enough for the page-move kernel's 32-bit chunk arithmetic.
bool small_pages(const dhs_pool* p) {
  return (int64_t)p->cfg.page_rows * p->cfg.row_bytes <= ((int64_t)1 << 24);
}

// Every call that enqueues device work starts here: the pool's device, and
// the pool's stream ordered after an outstanding dhs_prefetch.
int enter(dhs_pool* p) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return DHS_ECUDA;
  if (cur != p->device && cudaSetDevice(p->device) != cudaSuccess) return DHS_ECUDA;
  if (p->prefetch_pending) {
    if (cudaStreamWaitEvent(p->stream, p->ev_prefetch, 0) != cudaSuccess) return DHS_ECUDA;
    p->prefetch_pending = false;
    std::fill(p->pf_pair.begin(), p->pf_pair.end(), 0);
  }
  if (!p->join_gathers) return DHS_OK;
  for (cudaEvent_t e : p->ev_gathers) {
    if (cudaStreamWaitEvent(p->stream, e, 0) != cudaSuccess) return DHS_ECUDA;
    p->ev_free.push_back(e);
  }
  p->ev_gathers.clear();
  return DHS_OK;
}

// enter() for a resolve or gather of `st`: the outstanding prefetch is
// joined only if the step touches one of its pairs (a gather-only item may
// read any pair's rows, so it always joins); a step on other pairs runs
// alongside it -- their metadata, hot slots and miss lists are disjoint.
int enter_step(dhs_pool* p, const dhs_step* st) {
  // pending page copies or map uploads (the flush that follows) also join
  bool join = p->any_pending || p->dirty_hi >= 0;
  if (p->prefetch_pending && !join) {
    const dhs_pool_config& c = p->cfg;
    for (int32_t i = 0; i < st->n_items && !join; ++i) {
      const dhs_item& it = st->items[i];
      join = (it.flags & DHS_ITEM_GATHER_ONLY) ||
             p->pf_pair[(size_t)it.req * c.sources + it.src];
    }
  }
  if (join) return enter(p);
  const bool pending = p->prefetch_pending;
  p->prefetch_pending = false;  // device selection only
  const int rc = enter(p);
  p->prefetch_pending = pending;
  return rc;
}

void mark_dirty(dhs_pool* p, int64_t pair) {
  p->dirty_lo = std::min(p->dirty_lo, pair);
  p->dirty_hi = std::max(p->dirty_hi, pair);
}

// Copy pending resident pages (coalescing runs of consecutive pages in
// consecutive slots) and upload changed page maps, in stream order.
int flush(dhs_pool* p) {
  const dhs_pool_config& c = p->cfg;
  const size_t page_bytes = (size_t)c.page_rows * c.row_bytes;
  if (p->any_pending) {
    p->moves.clear();
    for (int64_t pair = 0; pair < p->pairs; ++pair) {
      PairState& s = p->ps[pair];
      if (s.pending.empty()) continue;
      std::sort(s.pending.begin(), s.pending.end());
      const int32_t* pm = p->map_host.data() + pair * p->pmax;
      if (!small_pages(p)) {  // pages too large for the page kernel: copy runs
        size_t i = 0;
        while (i < s.pending.size()) {
          const int32_t page = s.pending[i];
          const int32_t slot = pm[page];
          size_t run = 1;
          while (i + run < s.pending.size() && s.pending[i + run] == page + (int32_t)run &&
                 pm[page + run] == slot + (int32_t)run)
            ++run;
          cudaError_t e = cudaMemcpyAsync((uint8_t*)c.opt_dev + (size_t)slot * page_bytes,
                                          s.host + (size_t)page * page_bytes, run * page_bytes,
                                          cudaMemcpyHostToDevice, p->stream);
          if (e != cudaSuccess) return DHS_ECUDA;
          i += run;
        }
      } else {
        for (int32_t page : s.pending)
          p->moves.push_back({s.host_dev + (size_t)page * page_bytes,
                              (uint8_t*)c.opt_dev + (size_t)pm[page] * page_bytes});
      }
      s.pending.clear();
    }
    p->any_pending = false;
    if (!p->moves.empty() &&
        dhs::launch_page_moves(p->moves.data(), (int)p->moves.size(), (int)page_bytes,
                               2 * std::max(1, p->sm_count), p->stream) != cudaSuccess)
      return DHS_ECUDA;
  }
  if (p->dirty_hi >= 0) {
    const size_t off = (size_t)p->dirty_lo * p->pmax;
    const size_t cnt = (size_t)(p->dirty_hi - p->dirty_lo + 1) * p->pmax;
    cudaError_t e = cudaMemcpyAsync(p->map + off, p->map_host.data() + off, cnt * 4,
                                    cudaMemcpyHostToDevice, p->stream);
    if (e != cudaSuccess) return DHS_ECUDA;
    p->dirty_lo = INT64_MAX;
    p->dirty_hi = -1;
  }
  return DHS_OK;
}

void free_slot(dhs_pool* p, int64_t slot) {
  p->slot_pair[slot] = -1;
  p->slot_page[slot] = -1;
  p->used -= 1;
  if (slot < p->first_free) p->first_free = slot;
}

int64_t lowest_free_slot(dhs_pool* p) {
  for (int64_t i = p->first_free; i < p->cfg.optional_pages; ++i)
    if (p->slot_pair[i] < 0) {
      p->first_free = i;
      return i;
    }
  return -1;
}

// Free every optional page of pair; returns pages freed.
// Queue the device-to-host copy of one resident page whose backup was
// deferred (p->moves; launched by run_moves) and mark it backed.
int backup_page(dhs_pool* p, int64_t pair, int64_t q) {
  PairState& s = p->ps[pair];
  const dhs_pool_config& c = p->cfg;
  const size_t page_bytes = (size_t)c.page_rows * c.row_bytes;
  const int32_t slot = p->map_host[pair * p->pmax + q];
  const uint8_t* from = (const uint8_t*)c.opt_dev + (size_t)slot * page_bytes;
  if (small_pages(p)) {
    p->moves.push_back({from, s.host_dev + (size_t)q * page_bytes});
  } else if (cudaMemcpyAsync(s.host + (size_t)q * page_bytes, from, page_bytes,
                             cudaMemcpyDeviceToHost, p->stream) != cudaSuccess) {
    return DHS_ECUDA;
  }
  p->backup_order.erase({s.backup[q], pair * p->pmax + q});
  s.backup[q] = 0;
  return DHS_OK;
}

// Launch the queued page moves (in stream order, before anything enqueued
// after this call -- in particular before a freed slot is written again).
int run_moves(dhs_pool* p) {
  if (p->moves.empty()) return DHS_OK;
  const int pb = (int)((int64_t)p->cfg.page_rows * p->cfg.row_bytes);
  cudaError_t e = dhs::launch_page_moves(p->moves.data(), (int)p->moves.size(), pb,
                                         2 * std::max(1, p->sm_count), p->stream);
  p->moves.clear();
  return e == cudaSuccess ? DHS_OK : DHS_ECUDA;
}

// Free every optional page of pair; returns pages freed, or a negative DHS
// code.  backup: pages whose host backup is still deferred are backed up
// first (reclaim); a released request's pages need none.
int64_t drop_pages(dhs_pool* p, int64_t pair, bool backup) {
  int32_t* pm = p->map_host.data() + pair * p->pmax;
  PairState& s = p->ps[pair];
  int64_t n = 0;
  for (int64_t q = 0; q < p->pmax; ++q) {
    if (pm[q] < 0) continue;
    if (!s.backup.empty() && s.backup[q]) {
      if (backup) {
        const int rc = backup_page(p, pair, q);
        if (rc) return rc;
      } else {
        p->backup_order.erase({s.backup[q], pair * p->pmax + q});
        s.backup[q] = 0;
      }
    }
    free_slot(p, pm[q]);
    pm[q] = -1;
    ++n;
  }
  if (n) mark_dirty(p, pair);
  s.pending.clear();
  return n;
}

int64_t request_pages(const dhs_pool* p, int32_t r) {
  int64_t n = 0;
  for (int32_t s = 0; s < p->cfg.sources; ++s) {
    const int32_t* pm = p->map_host.data() + ((int64_t)r * p->cfg.sources + s) * p->pmax;
    for (int64_t q = 0; q < p->pmax; ++q) n += pm[q] >= 0;
  }
  return n;
}

}  // namespace

extern "C" {

const char* dhs_strerror(int code) {
  switch (code) {
    case DHS_OK: return "ok";
    case DHS_EINVAL: return "invalid argument";
    case DHS_ENOMEM: return "out of host memory";
    case DHS_EWOULDWAIT: return "capacity deficit: admission waits";
    case DHS_EBUDGET: return "more missing rows than unprotected hot slots";
    case DHS_ERANGE: return "row or location out of range";
    case DHS_ETIMEDOUT: return "bounded device wait gave up";
    case DHS_ECUDA: return "CUDA runtime error";
    case DHS_ESTATE: return "request/source not admitted or already admitted";
    default: return "unknown error";
  }
}

int dhs_pool_bytes(const dhs_pool_config* cfg, size_t out[DHS_NUM_BUFS]) {
  int rc = validate_geometry(cfg);
  if (rc) return rc;
  if (!out) return DHS_EINVAL;
  const size_t pairs = (size_t)cfg->max_requests * cfg->sources;
  out[DHS_BUF_HOT] = pairs * cfg->hot_rows * (size_t)cfg->row_bytes;
  out[DHS_BUF_TAIL] = pairs * cfg->tail_rows * (size_t)cfg->row_bytes;
  out[DHS_BUF_OPT] = (size_t)cfg->optional_pages * cfg->page_rows * (size_t)cfg->row_bytes;
  out[DHS_BUF_META] = meta_layout(*cfg).total;
  return DHS_OK;
}

int dhs_pool_create(const dhs_pool_config* cfg, dhs_pool** out) {
  if (!out) return DHS_EINVAL;
  *out = nullptr;
  int rc = validate_geometry(cfg);
  if (rc) return rc;
  auto aligned = [](const void* q) { return q && ((uintptr_t)q % kAlign) == 0; };
  if (!aligned(cfg->hot_dev) || !aligned(cfg->tail_dev) || !aligned(cfg->meta_dev))
    return DHS_EINVAL;
  if (cfg->optional_pages > 0 && !aligned(cfg->opt_dev)) return DHS_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DHS_ECUDA;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return DHS_ECUDA;
  int sms = 0, smem_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess)
    return DHS_ECUDA;
  const size_t smem = max_resolve_smem(*cfg, false);
  if (smem + 1024 > (size_t)optin) return DHS_EINVAL;
  const size_t smem_u = max_resolve_smem(*cfg, true);
  const bool union_ok = smem_u + 1024 <= (size_t)optin;
  if (dhs::resolve_set_smem_limit(union_ok ? smem_u : smem) != cudaSuccess) return DHS_ECUDA;

  dhs_pool* p = new (std::nothrow) dhs_pool();
  if (!p) return DHS_ENOMEM;
  try {
    p->cfg = *cfg;
    p->union_ok = union_ok;
    p->gather_impl = dhs::kGatherTma;
    p->sm_count = sms;
    p->smem_optin = optin;
    p->smem_per_sm = smem_sm;
    p->stream = (cudaStream_t)cfg->stream;
    p->device = dev;
    p->pairs = (int64_t)cfg->max_requests * cfg->sources;
    p->pmax = pages_max_of(*cfg);
    p->mcap = mcap_of(*cfg);
    p->page_shift = log2i(cfg->page_rows);
    p->layout = meta_layout(*cfg);
    uint8_t* m = (uint8_t*)cfg->meta_dev;
    p->tags = (int32_t*)(m + p->layout.tags);
    p->stamps = (uint32_t*)(m + p->layout.stamps);
    p->map = (int32_t*)(m + p->layout.map);
    p->miss_rows = (int32_t*)(m + p->layout.miss_rows);
    p->miss_slots = (int32_t*)(m + p->layout.miss_slots);
    p->miss_count = (uint32_t*)(m + p->layout.miss_count);
    p->copy_cursor = (uint32_t*)(m + p->layout.copy_cursor);
    p->pair_status = (int32_t*)(m + p->layout.pair_status);
    p->loc_ready = (uint32_t*)(m + p->layout.loc_ready);
    p->copy_ready = (uint32_t*)(m + p->layout.copy_ready);
    p->fill = (uint32_t*)(m + p->layout.fill);
    p->later_count = (uint32_t*)(m + p->layout.later_count);
    p->later = (dhs::LaterEntry*)(m + p->layout.later);
    p->later_cap = later_cap_of(*cfg);
    p->fill_words = (int)fill_words_of(*cfg);
    p->miss_off = (int32_t*)(m + p->layout.miss_off);
    p->miss_ent = (int32_t*)(m + p->layout.miss_ent);
    p->ent_cap = ent_cap_of(*cfg);
    p->status = (uint32_t*)(m + p->layout.status);
    p->ps.resize(p->pairs);
    p->map_host.assign((size_t)(p->pairs * p->pmax), -1);
    p->slot_pair.assign((size_t)cfg->optional_pages + 1, -1);
    p->slot_page.assign((size_t)cfg->optional_pages + 1, -1);
    p->seen.assign((size_t)p->pairs, 0);
    p->app_of_pair.assign((size_t)p->pairs, -1);
    p->l0_of_pair.assign((size_t)p->pairs, 0);
    p->app_of_pair_rows.assign((size_t)p->pairs, nullptr);
    p->seq_of_pair.assign((size_t)p->pairs, 0);
    p->pf_pair.assign((size_t)p->pairs, 0);
    p->staged_pair.assign((size_t)p->pairs, 0);
  } catch (...) {
    delete p;
    return DHS_ENOMEM;
  }
  if (dhs::resolve_set_carveout() != cudaSuccess ||
      dhs::hostcopy_set_carveout(copy_hold_limit(optin)) != cudaSuccess ||
      dhs::gather_set_carveout() != cudaSuccess || dhs::append_set_carveout() != cudaSuccess) {
    delete p;
    return DHS_ECUDA;
  }
  if (dhs::gather_set_smem_limit(cfg->row_bytes, optin, &p->tma_ok) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_main, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_prefetch, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&p->ev_step, cudaEventDisableTiming) != cudaSuccess) {
    delete p;
    return DHS_ECUDA;
  }
  if (!p->tma_ok) p->gather_impl = dhs::kGatherVector;  // rows too large to stage a tile
  // empty hot caches (tag -1, stamp 0), no ready pages, zero counts/status
  cudaError_t e = cudaMemsetAsync(p->tags, 0xFF, p->pairs * cfg->hot_rows * 4, p->stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(p->stamps, 0, p->pairs * cfg->hot_rows * 4, p->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->map, 0xFF, p->pairs * p->pmax * 4, p->stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync((uint8_t*)cfg->meta_dev + p->layout.miss_count, 0,
                        p->layout.later - p->layout.miss_count, p->stream);
  if (e != cudaSuccess) {
    delete p;
    return DHS_ECUDA;
  }
  *out = p;
  return DHS_OK;
}

void dhs_pool_destroy(dhs_pool* pool) { delete pool; }

int64_t dhs_pool_used(const dhs_pool* pool) { return pool ? pool->used : -1; }

int dhs_set_option(dhs_pool* pool, int32_t key, int64_t value) {
  if (!pool) return DHS_EINVAL;
  if (key == DHS_OPT_COPY_CTAS) {
    if (value < 0 || value > 4096) return DHS_EINVAL;
    pool->copy_ctas = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_TRACE) {
    if (value < 0 || (value & 7)) return DHS_EINVAL;
    pool->trace = (unsigned long long*)(uintptr_t)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_EARLY) {
    if (value < 0 || value > 1) return DHS_EINVAL;
    pool->early = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_GATHER_IMPL) {
    if (value != dhs::kGatherVector && !(value == dhs::kGatherTma && pool->tma_ok))
      return DHS_EINVAL;
    pool->gather_impl = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_FRESH_LIST) {
    if (value < -1 || value > 1) return DHS_EINVAL;
    pool->fresh_list = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_STAGE_MISSES) {
    if (value < 0 || value > 1) return DHS_EINVAL;
    pool->stage_misses = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_GATHER_TPC) {
    if (value < 1 || value > 64) return DHS_EINVAL;
    pool->gather_tpc = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_RESOLVE_PAIRED) {
    if (value < -1 || value > 1) return DHS_EINVAL;
    pool->resolve_paired = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_COPY_PDL) {
    if (value < -1 || value > 1) return DHS_EINVAL;
    pool->copy_pdl = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_COPY_STEAL) {
    if (value < -1 || value > 1) return DHS_EINVAL;
    pool->copy_steal = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_RESOLVE_CTAS) {
    if (value < 0 || value > (1 << 20)) return DHS_EINVAL;
    pool->resolve_ctas = (int)value;
    return DHS_OK;
  }
  if (key == DHS_OPT_MARK_POLLS) {
    if (value < -1 || value > (int64_t)dhs::kMarkPolls) return DHS_EINVAL;
    pool->mark_polls = value < 0 ? dhs::kMarkPolls : (uint32_t)value;
    return DHS_OK;
  }
  return DHS_EINVAL;
}

// Whether fused steps hand fresh rows to the list copied after the host-copy
// grid (one launch more per step).  Auto: when more than a tenth of the
// admitted complete pages are not optional-resident, so that host copies are
// expected every step.
static bool tma_gather(const dhs_pool* p) { return p->gather_impl == dhs::kGatherTma; }

static bool use_fresh_list(const dhs_pool* p) {
  if (!tma_gather(p) || !p->early) return false;
  if (p->fresh_list >= 0) return p->fresh_list == 1;
  return (p->complete_pages - p->used) * 10 > p->complete_pages;
}

int dhs_get_option(dhs_pool* pool, int32_t key, int64_t* value) {
  if (!pool || !value) return DHS_EINVAL;
  switch (key) {
    case DHS_OPT_COPY_CTAS: *value = pool->copy_ctas; return DHS_OK;
    case DHS_OPT_GATHER_IMPL: *value = pool->gather_impl; return DHS_OK;
    case DHS_OPT_TRACE: *value = (int64_t)(uintptr_t)pool->trace; return DHS_OK;
    case DHS_OPT_EARLY: *value = pool->early; return DHS_OK;
    case DHS_OPT_FRESH_LIST: *value = use_fresh_list(pool) ? 1 : 0; return DHS_OK;
    case DHS_OPT_GATHER_TPC: *value = pool->gather_tpc; return DHS_OK;
    case DHS_OPT_STAGE_MISSES: *value = pool->stage_misses; return DHS_OK;
    case DHS_OPT_MARK_POLLS: *value = pool->mark_polls; return DHS_OK;
    case DHS_OPT_COPY_PDL: *value = pool->copy_pdl; return DHS_OK;
    case DHS_OPT_RESOLVE_PAIRED: *value = pool->resolve_paired; return DHS_OK;
    case DHS_OPT_COPY_STEAL: *value = pool->copy_steal; return DHS_OK;
    case DHS_OPT_RESOLVE_CTAS: *value = pool->resolve_ctas; return DHS_OK;
    default: return DHS_EINVAL;
  }
}

int dhs_admit(dhs_pool* p, int32_t req, int32_t src, void* host_rows, int64_t n_rows,
              const uint8_t* mask, int64_t* deficit) {
  if (deficit) *deficit = 0;
  if (!p || req < 0 || req >= p->cfg.max_requests || src < 0 || src >= p->cfg.sources)
    return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  if (n_rows < 0 || n_rows > c.max_rows_per_request || !host_rows) return DHS_EINVAL;
  if ((uintptr_t)host_rows % 16) return DHS_EINVAL;  // rows move in 16-byte chunks
  const int64_t pair = (int64_t)req * c.sources + src;
  PairState& s = p->ps[pair];
  if (s.admitted) return DHS_ESTATE;
  int rc = enter(p);
  if (rc) return rc;
  void* hdev = nullptr;
  if (cudaHostGetDevicePointer(&hdev, host_rows, 0) != cudaSuccess || !hdev ||
      (uintptr_t)hdev % 16) {
    cudaGetLastError();  // clear the sticky-free error state
    return DHS_EINVAL;
  }
  const int64_t complete = n_rows / c.page_rows;
  int64_t want = 0;
  for (int64_t q = 0; q < complete; ++q) want += (!mask || mask[q]) ? 1 : 0;
  const int64_t usable = c.optional_pages - c.admission_reserve_pages;
  if (p->used + want > usable) {
    if (deficit) *deficit = p->used + want - usable;
    return DHS_EWOULDWAIT;
  }
  // tail ring <- rows [max(0, N-T), N)
  const int64_t T = c.tail_rows, rb = c.row_bytes;
  const int64_t lo = std::max<int64_t>(0, n_rows - T);
  int64_t row = lo;
  while (row < n_rows) {
    const int64_t slot = row % T;
    const int64_t run = std::min(n_rows - row, T - slot);
    cudaError_t e = cudaMemcpyAsync((uint8_t*)c.tail_dev + ((size_t)pair * T + slot) * rb,
                                    (uint8_t*)host_rows + (size_t)row * rb, run * rb,
                                    cudaMemcpyHostToDevice, p->stream);
    if (e != cudaSuccess) return DHS_ECUDA;
    row += run;
  }
  int32_t* pm = p->map_host.data() + pair * p->pmax;
  for (int64_t q = 0; q < complete; ++q) {
    if (mask && !mask[q]) continue;
    const int64_t slot = lowest_free_slot(p);
    p->slot_pair[slot] = (int32_t)pair;
    p->slot_page[slot] = (int32_t)q;
    p->used += 1;
    pm[q] = (int32_t)slot;
    s.pending.push_back((int32_t)q);
  }
  if (want) {
    p->any_pending = true;
    mark_dirty(p, pair);
  }
  s.admitted = true;
  s.N = n_rows;
  s.L = n_rows;
  p->complete_pages += n_rows >> p->page_shift;
  s.host = (uint8_t*)host_rows;
  s.host_dev = (uint8_t*)hdev;
  return DHS_OK;
}

int dhs_admit_device(dhs_pool* p, int32_t req, int32_t src, const void* dev_rows,
                     void* host_rows, int64_t n_rows, const uint8_t* mask,
                     int64_t* deficit) {
  if (deficit) *deficit = 0;
  if (!p || req < 0 || req >= p->cfg.max_requests || src < 0 || src >= p->cfg.sources)
    return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  if (n_rows < 0 || n_rows > c.max_rows_per_request || !host_rows) return DHS_EINVAL;
  if (n_rows > 0 && !dev_rows) return DHS_EINVAL;
  if ((uintptr_t)host_rows % 16) return DHS_EINVAL;
  const int64_t pair = (int64_t)req * c.sources + src;
  PairState& s = p->ps[pair];
  if (s.admitted) return DHS_ESTATE;
  int rc = enter(p);
  if (rc) return rc;
  void* hdev = nullptr;
  if (cudaHostGetDevicePointer(&hdev, host_rows, 0) != cudaSuccess || !hdev ||
      (uintptr_t)hdev % 16) {
    cudaGetLastError();
    return DHS_EINVAL;
  }
  const int64_t complete = n_rows / c.page_rows;
  int64_t want = 0;
  for (int64_t q = 0; q < complete; ++q) want += (!mask || mask[q]) ? 1 : 0;
  const int64_t usable = c.optional_pages - c.admission_reserve_pages;
  if (p->used + want > usable) {
    if (deficit) *deficit = p->used + want - usable;
    return DHS_EWOULDWAIT;
  }
  // the copies are enqueued now; the page map reaches the device at the next
  // flush, after them in stream order
  const int64_t T = c.tail_rows, rb = c.row_bytes, PR = c.page_rows;
  const size_t page_bytes = (size_t)PR * rb;
  const uint8_t* dsrc = (const uint8_t*)dev_rows;
  uint8_t* hdst = (uint8_t*)host_rows;
  auto copy = [&](void* dst, const void* from, size_t bytes, cudaMemcpyKind kind) {
    return cudaMemcpyAsync(dst, from, bytes, kind, p->stream) == cudaSuccess;
  };
  // tail ring <- rows [max(0, N-T), N)
  for (int64_t row = std::max<int64_t>(0, n_rows - T); row < n_rows;) {
    const int64_t slot = row % T;
    const int64_t run = std::min(n_rows - row, T - slot);
    if (!copy((uint8_t*)c.tail_dev + ((size_t)pair * T + slot) * rb, dsrc + (size_t)row * rb,
              run * rb, cudaMemcpyDeviceToDevice))
      return DHS_ECUDA;
    row += run;
  }
  int32_t* pm = p->map_host.data() + pair * p->pmax;
  s.backup.assign((size_t)p->pmax, 0);
  for (int64_t q = 0; q < complete; ++q) {
    if (mask && !mask[q]) continue;
    const int64_t slot = lowest_free_slot(p);
    p->slot_pair[slot] = (int32_t)pair;
    p->slot_page[slot] = (int32_t)q;
    p->used += 1;
    pm[q] = (int32_t)slot;
    s.backup[q] = ++p->bseq;
    p->backup_order.insert({s.backup[q], pair * p->pmax + q});
  }
  // resident pages: device to device, runs of consecutive pages and slots;
  // every other imported row: device to host now, runs of consecutive rows
  for (int64_t q = 0; q < complete;) {
    int64_t run = 1;
    if (pm[q] >= 0) {
      while (q + run < complete && pm[q + run] == pm[q] + run) ++run;
      if (!copy((uint8_t*)c.opt_dev + (size_t)pm[q] * page_bytes, dsrc + q * page_bytes,
                run * page_bytes, cudaMemcpyDeviceToDevice))
        return DHS_ECUDA;
    } else {
      while (q + run < complete && pm[q + run] < 0) ++run;
      if (!copy(hdst + q * page_bytes, dsrc + q * page_bytes, run * page_bytes,
                cudaMemcpyDeviceToHost))
        return DHS_ECUDA;
    }
    q += run;
  }
  if (n_rows > complete * PR &&
      !copy(hdst + complete * page_bytes, dsrc + complete * page_bytes,
            (size_t)(n_rows - complete * PR) * rb, cudaMemcpyDeviceToHost))
    return DHS_ECUDA;
  if (want) mark_dirty(p, pair);
  s.admitted = true;
  s.N = n_rows;
  s.L = n_rows;
  p->complete_pages += complete;
  s.host = (uint8_t*)host_rows;
  s.host_dev = (uint8_t*)hdev;
  return DHS_OK;
}

int dhs_backup(dhs_pool* p, int64_t max_pages, int64_t* done) {
  if (done) *done = 0;
  if (!p || max_pages < 0) return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  p->moves.clear();
  int64_t n = 0;
  while (n < max_pages && !p->backup_order.empty()) {
    const int64_t key = p->backup_order.begin()->second;
    if ((rc = backup_page(p, key / p->pmax, key % p->pmax))) return rc;
    ++n;
  }
  if ((rc = run_moves(p))) return rc;
  if (done) *done = n;
  return DHS_OK;
}

int dhs_admit_window(dhs_pool* p, int32_t req, int32_t src, const void* dev_rows,
                     int64_t n_rows) {
  if (!p || req < 0 || req >= p->cfg.max_requests || src < 0 || src >= p->cfg.sources)
    return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  if (n_rows < 0 || n_rows > c.max_rows_per_request) return DHS_EINVAL;
  if (n_rows > 0 && (!dev_rows || (uintptr_t)dev_rows % 16)) return DHS_EINVAL;
  const int64_t pair = (int64_t)req * c.sources + src;
  PairState& s = p->ps[pair];
  if (s.admitted) return DHS_ESTATE;
  int rc = enter(p);
  if (rc) return rc;
  // the window's rows [N - m, N) into ring slots row mod T (at most two runs)
  const int64_t T = c.tail_rows, rb = c.row_bytes;
  const int64_t m = std::min<int64_t>(n_rows, T);
  for (int64_t row = n_rows - m; row < n_rows;) {
    const int64_t slot = row % T;
    const int64_t run = std::min(n_rows - row, T - slot);
    cudaError_t e = cudaMemcpyAsync((uint8_t*)c.tail_dev + ((size_t)pair * T + slot) * rb,
                                    (const uint8_t*)dev_rows + (size_t)(row - (n_rows - m)) * rb,
                                    run * rb, cudaMemcpyDeviceToDevice, p->stream);
    if (e != cudaSuccess) return DHS_ECUDA;
    row += run;
  }
  s.admitted = true;
  s.window = true;
  s.N = 0;  // no imported pages: nothing for the optional map, refill or reclaim
  s.L = n_rows;
  return DHS_OK;
}

int64_t dhs_pending_backup(const dhs_pool* p) {
  return p ? (int64_t)p->backup_order.size() : -1;
}

int dhs_refill(dhs_pool* p, int64_t max_pages, int64_t* filled) {
  if (filled) *filled = 0;
  if (!p || max_pages < 0) return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  const int64_t usable = c.optional_pages - c.admission_reserve_pages;
  int64_t n = 0, idle = 0;
  int32_t r = p->rr;
  while (n < max_pages && p->used < usable && idle < c.max_requests) {
    bool found = false;
    for (int32_t src = 0; src < c.sources && !found; ++src) {
      const int64_t pair = (int64_t)r * c.sources + src;
      PairState& s = p->ps[pair];
      if (!s.admitted) continue;
      int32_t* pm = p->map_host.data() + pair * p->pmax;
      for (int64_t q = 0; q < s.N / c.page_rows && !found; ++q) {
        if (pm[q] >= 0) continue;
        const int64_t slot = lowest_free_slot(p);
        p->slot_pair[slot] = (int32_t)pair;
        p->slot_page[slot] = (int32_t)q;
        p->used += 1;
        pm[q] = (int32_t)slot;
        s.pending.push_back((int32_t)q);  // copied from the host copy at flush
        p->any_pending = true;
        mark_dirty(p, pair);
        found = true;
      }
    }
    if (found) {
      ++n;
      idle = 0;
    } else {
      ++idle;
    }
    r = (r + 1) % c.max_requests;
  }
  p->rr = r;
  if (filled) *filled = n;
  return DHS_OK;
}

int dhs_reclaim(dhs_pool* p, const int32_t* order, int32_t n, int64_t deficit,
                int64_t* freed) {
  if (freed) *freed = 0;
  if (!p || n < 0 || deficit < 0 || (n > 0 && !order)) return DHS_EINVAL;
  for (int32_t i = 0; i < n; ++i)
    if (order[i] < 0 || order[i] >= p->cfg.max_requests) return DHS_EINVAL;
  int64_t avail = 0;
  std::vector<uint8_t> counted((size_t)p->cfg.max_requests, 0);
  for (int32_t i = 0; i < n; ++i) {
    if (counted[order[i]]) continue;
    counted[order[i]] = 1;
    avail += request_pages(p, order[i]);
  }
  if (avail < deficit) return DHS_EWOULDWAIT;
  int rc = enter(p);
  if (rc) return rc;
  p->moves.clear();
  int64_t got = 0;
  for (int32_t i = 0; i < n && got < deficit; ++i)
    for (int32_t s = 0; s < p->cfg.sources; ++s) {
      const int64_t k = drop_pages(p, (int64_t)order[i] * p->cfg.sources + s, true);
      if (k < 0) return (int)k;
      got += k;
    }
  if ((rc = run_moves(p))) return rc;  // backups before any reuse of the slots
  if (freed) *freed = got;
  return DHS_OK;
}

int dhs_release(dhs_pool* p, int32_t req) {
  if (!p || req < 0 || req >= p->cfg.max_requests) return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  const int64_t B = p->cfg.hot_rows;
  for (int32_t s = 0; s < p->cfg.sources; ++s) {
    const int64_t pair = (int64_t)req * p->cfg.sources + s;
    drop_pages(p, pair, false);
    if (p->ps[pair].admitted) p->complete_pages -= p->ps[pair].N >> p->page_shift;
    p->ps[pair] = PairState();
  }
  const int64_t pair0 = (int64_t)req * p->cfg.sources;
  cudaError_t e = cudaMemsetAsync(p->tags + pair0 * B, 0xFF, p->cfg.sources * B * 4, p->stream);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(p->stamps + pair0 * B, 0, p->cfg.sources * B * 4, p->stream);
  return cuda_rc(e);
}

int dhs_flush(dhs_pool* p) {
  if (!p) return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  return flush(p);
}

int dhs_append(dhs_pool* p, const dhs_append_item* items, int32_t n_items) {
  if (!p || n_items < 0 || (n_items > 0 && !items)) return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  std::fill(p->seen.begin(), p->seen.end(), 0);
  for (int32_t i = 0; i < n_items; ++i) {
    const dhs_append_item& it = items[i];
    if (it.req < 0 || it.req >= c.max_requests || it.src < 0 || it.src >= c.sources)
      return DHS_EINVAL;
    if (it.count < 0 || it.count > c.tail_rows) return DHS_EINVAL;
    if (it.count > 0 && !it.rows_dev) return DHS_EINVAL;
    const int64_t pair = (int64_t)it.req * c.sources + it.src;
    if (p->seen[pair]) return DHS_EINVAL;
    p->seen[pair] = 1;
    const PairState& s = p->ps[pair];
    if (!s.admitted) return DHS_ESTATE;
    if (s.L + it.count > c.max_rows_per_request) return DHS_EINVAL;
  }
  int rc = enter(p);
  if (rc) return rc;
  p->aitems.clear();
  for (int32_t i = 0; i < n_items; ++i) {
    const dhs_append_item& it = items[i];
    if (it.count == 0) continue;
    const int64_t pair = (int64_t)it.req * c.sources + it.src;
    PairState& s = p->ps[pair];
    dhs::AppendItem a;
    a.rows = (const uint8_t*)it.rows_dev;
    a.host = s.host_dev;
    a.L0 = s.L;
    a.pair = (int32_t)pair;
    a.count = it.count;
    p->aitems.push_back(a);
    s.L += it.count;
  }
  dhs::AppendCommon ac{};
  ac.tail = (uint8_t*)c.tail_dev;
  ac.T = c.tail_rows;
  ac.row_bytes = c.row_bytes;
  for (size_t b = 0; b < p->aitems.size(); b += dhs::kAppendItemsMax) {
    const int n = (int)std::min<size_t>(dhs::kAppendItemsMax, p->aitems.size() - b);
    if (dhs::launch_append(ac, p->aitems.data() + b, n, p->stream) != cudaSuccess)
      return DHS_ECUDA;
  }
  return DHS_OK;
}

static int validate_step(dhs_pool* p, const dhs_step* st, bool resolving) {
  if (!p || !st || st->n_items < 0 || (st->n_items > 0 && !st->items)) return DHS_EINVAL;
  if (resolving && st->step == 0) return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  if (resolving) std::fill(p->seen.begin(), p->seen.end(), 0);
  for (int32_t i = 0; i < st->n_items; ++i) {
    const dhs_item& it = st->items[i];
    if (it.queries < 0 || it.topk < 0) return DHS_EINVAL;
    const int64_t n = (int64_t)it.queries * it.topk;
    if (n > INT32_MAX) return DHS_EINVAL;
    if (n > 0 && !it.loc_dev) return DHS_EINVAL;
    if (!resolving) {
      if (n > 0 && !it.staging_dev) return DHS_EINVAL;
      continue;
    }
    if (it.flags & DHS_ITEM_GATHER_ONLY) continue;
    if (it.queries > c.max_queries || it.topk > c.max_topk) return DHS_EINVAL;
    if (it.req < 0 || it.req >= c.max_requests || it.src < 0 || it.src >= c.sources)
      return DHS_EINVAL;
    if (n > 0 && !it.sel_dev) return DHS_EINVAL;
    if ((it.flags & DHS_ITEM_UNION) && (!p->union_ok || (n > 0 && !it.index_dev)))
      return DHS_EINVAL;
    const int64_t pair = (int64_t)it.req * c.sources + it.src;
    if (p->seen[pair]) return DHS_EINVAL;
    p->seen[pair] = 1;
    if (!p->ps[pair].admitted) return DHS_ESTATE;
  }
  return DHS_OK;
}

// Launch resolve + host copy for every resolving item of a validated,
// flushed step.  `apps` (may be null): appends folded into the resolve
// kernel, one per pair listed in p->app_of_pair.
static int resolve_impl(dhs_pool* p, const dhs_step* st, const dhs_append_item* apps,
                        bool fused, const dhs::NoallocScratch* scr = nullptr) {
  const dhs_pool_config& c = p->cfg;
  p->ritems.clear();
  p->citems.clear();
  for (int32_t i = 0; i < st->n_items; ++i) {
    const dhs_item& it = st->items[i];
    if (it.flags & DHS_ITEM_GATHER_ONLY) continue;
    const int64_t pair = (int64_t)it.req * c.sources + it.src;
    PairState& s = p->ps[pair];
    dhs::ResolveItem r{};
    p->l0_of_pair[pair] = s.L;
    p->app_of_pair_rows[pair] = nullptr;
    if (apps && p->app_of_pair[pair] >= 0) {
      const dhs_append_item& a = apps[p->app_of_pair[pair]];
      r.app_rows = (const uint8_t*)a.rows_dev;
      r.app_host = s.host_dev;
      r.app_L0 = s.L;
      r.app_count = a.count;
      s.L += a.count;
      p->app_of_pair_rows[pair] = (const uint8_t*)a.rows_dev;
    }
    r.sel = it.sel_dev;
    r.loc = it.loc_dev;
    r.counters = it.counters_dev;
    r.index = (it.flags & DHS_ITEM_UNION) ? it.index_dev : nullptr;
    r.L = s.L;
    r.N = s.N;
    r.lo = s.window ? std::max<int64_t>(0, s.L - c.tail_rows) : 0;
    r.pair = (int32_t)pair;
    r.n = it.queries * it.topk;
    // fused steps: the host copy writes the misses into the item's staging,
    // and its gather leaves them out
    const bool stage = fused && !scr && p->stage_misses && tma_gather(p) && p->early &&
                       it.staging_dev != nullptr && r.n > 0;
    r.stage = stage ? 1 : 0;
    p->staged_pair[pair] = stage ? 1 : 0;
    p->ritems.push_back(r);
    dhs::CopyItem ci{};
    ci.host = s.host_dev;
    ci.staging = stage ? (uint8_t*)it.staging_dev : nullptr;
    ci.pair = (int32_t)pair;
    p->citems.push_back(ci);
  }
  // gather-only (Reuse) items handed a resolved item's location vector: the
  // resolved item publishes its locations for them, and when it is staged
  // with the same entries, the host copy writes their fetched rows too
  p->staged_item.assign((size_t)st->n_items, 0);
  for (int32_t i = 0; i < st->n_items; ++i) {
    const dhs_item& it = st->items[i];
    if (!(it.flags & DHS_ITEM_GATHER_ONLY) || !it.loc_dev) continue;
    bool first = true;
    for (size_t k = 0; k < p->ritems.size(); ++k) {
      dhs::CopyItem& ci = p->citems[k];
      if (p->ritems[k].loc != it.loc_dev) continue;
      p->ritems[k].loc_shared = 1;
      if (first && it.staging_dev && ci.staging && p->ritems[k].n == it.queries * it.topk &&
          ci.nshare < dhs::kCopyShareMax) {
        ci.share[ci.nshare++] = (uint8_t*)it.staging_dev;
        p->staged_item[i] = 1;
      }
      first = false;
    }
  }
  dhs::ResolveCommon rcm{};
  rcm.tags = p->tags;
  rcm.stamps = p->stamps;
  rcm.map = p->map;
  // miss lists: the pool's metadata, or the fixed scratch of
  // dhs_resolve_noalloc
  rcm.miss_rows = scr ? scr->miss_rows : p->miss_rows;
  rcm.miss_slots = scr ? scr->miss_slots : p->miss_slots;
  rcm.miss_count = scr ? scr->miss_count : p->miss_count;
  rcm.copy_cursor = p->copy_cursor;
  rcm.pair_status = p->pair_status;
  rcm.status = p->status;
  rcm.T = c.tail_rows;
  rcm.B = c.hot_rows;
  rcm.Pmax = (int32_t)p->pmax;
  rcm.Mcap = (int32_t)p->mcap;
  rcm.page_shift = p->page_shift;
  rcm.step = st->step;
  rcm.row_bytes = c.row_bytes;
  rcm.tail = (uint8_t*)c.tail_dev;
  rcm.trace = p->trace;
  p->fused_resolved = fused && !p->ritems.empty();
  if (p->fused_resolved) ++p->gen;
  rcm.loc_ready = p->loc_ready;
  rcm.copy_ready = p->copy_ready;
  rcm.fill = p->fill;
  rcm.fill_words = p->fill_words;
  rcm.later_count = p->later_count;
  rcm.gen = p->gen;
  rcm.miss_off = p->miss_off;
  rcm.miss_ent = p->miss_ent;
  rcm.ent_cap = (int32_t)p->ent_cap;
  dhs::CopyCommon ccm{};
  ccm.hot = (uint8_t*)c.hot_dev;
  ccm.miss_rows = rcm.miss_rows;
  ccm.miss_slots = rcm.miss_slots;
  ccm.miss_count = rcm.miss_count;
  ccm.cursor = p->copy_cursor;
  ccm.miss_off = p->miss_off;
  ccm.miss_ent = p->miss_ent;
  ccm.ent_cap = (int32_t)p->ent_cap;
  ccm.B = c.hot_rows;
  ccm.Mcap = (int32_t)p->mcap;
  ccm.row_bytes = c.row_bytes;
  ccm.trace = p->trace;
  ccm.mark_polls = p->mark_polls;
  const size_t nr = p->ritems.size();
  for (size_t b = 0; b < nr; b += dhs::kResolveItemsLarge) {
    const int n = (int)std::min<size_t>(dhs::kResolveItemsLarge, nr - b);
    int64_t wmax = 0, qmax = 0, nmax = 0;
    bool uni = false;
    for (int i = 0; i < n; ++i) {
      const dhs::ResolveItem& r = p->ritems[b + i];
      uni |= r.index != nullptr;
      wmax = std::max<int64_t>(wmax, (r.L + 63) / 64);
      qmax = std::max<int64_t>(qmax, std::min<int64_t>(std::min<int64_t>(r.n, r.L), c.hot_rows));
      nmax = std::max<int64_t>(nmax, r.n);
    }
    rcm.w64cap = (int32_t)wmax;
    rcm.qkcap = (int32_t)qmax;
    rcm.seq = ++p->seq & dhs::kSeqMask;
    if (rcm.seq == 0) rcm.seq = p->seq = 1;  // 0 never matches a published mark
    ccm.ready = rcm.copy_ready;  // the copy starts on each item once its misses are listed
    ccm.seq = rcm.seq;
    for (int i = 0; i < n; ++i) p->seq_of_pair[p->ritems[b + i].pair] = rcm.seq;
    rcm.uni = uni ? 1 : 0;
    // stage the selections in shared memory when the plan leaves room for them
    const size_t base = dhs::resolve_smem_bytes(rcm.w64cap, rcm.qkcap, c.hot_rows, uni, 0);
    const size_t staged =
        dhs::resolve_smem_bytes(rcm.w64cap, rcm.qkcap, c.hot_rows, uni, (int)nmax);
    const bool paired = resolve_paired(p, n, base);
    const int threads = n <= dhs::kResolveItemsSmall
                            ? dhs::resolve_threads(dhs::kResolveItemsSmall)
                            : (paired ? dhs::kResolvePairThreads
                                      : dhs::resolve_threads(dhs::kResolveItemsLarge));
    rcm.selcap = 0;
    if (!paired && nmax >= 8 * threads && staged + 1024 <= (size_t)p->smem_optin &&
        dhs::resolve_set_smem_limit(staged) == cudaSuccess)
      rcm.selcap = (int32_t)nmax;
    const size_t smem = rcm.selcap ? staged : base;
    if (dhs::launch_resolve(rcm, p->ritems.data() + b, n, resolve_ctas(p, n, paired), smem,
                            paired, p->stream) !=
        cudaSuccess)
      return DHS_ECUDA;
    ccm.steal = copy_steal(p, n) ? 1 : 0;
    if (dhs::launch_hostcopy(ccm, p->citems.data() + b, n, copy_ctas(p, n), copy_threads(p, n),
                             copy_pdl(p, n), copy_hold_smem(p, n), p->stream) != cudaSuccess)
      return DHS_ECUDA;
  }
  return DHS_OK;
}

int dhs_prefetch(dhs_pool* p, const dhs_step* st, void* side_stream) {
  if (!p || !side_stream) return DHS_EINVAL;
  int rc = validate_step(p, st, true);
  if (rc) return rc;
  if ((rc = enter(p))) return rc;
  // pending page copies and map uploads, then everything the pool's stream
  // holds so far (earlier gathers still reading hot slots), come first
  if ((rc = flush(p))) return rc;
  cudaStream_t side = (cudaStream_t)side_stream;
  if (cudaEventRecord(p->ev_main, p->stream) != cudaSuccess ||
      cudaStreamWaitEvent(side, p->ev_main, 0) != cudaSuccess)
    return DHS_ECUDA;
  cudaStream_t main = p->stream;
  p->stream = side;
  rc = resolve_impl(p, st, nullptr, false);
  p->stream = main;
  // whatever was enqueued on the side stream is joined before the pool's next
  // device work, even if the call failed part way
  if (cudaEventRecord(p->ev_prefetch, side) != cudaSuccess) return DHS_ECUDA;
  p->prefetch_pending = true;
  for (int32_t i = 0; i < st->n_items; ++i) {
    const dhs_item& it = st->items[i];
    if (!(it.flags & DHS_ITEM_GATHER_ONLY))
      p->pf_pair[(size_t)it.req * p->cfg.sources + it.src] = 1;
  }
  return rc;
}

int dhs_resolve(dhs_pool* p, const dhs_step* st) {
  int rc = validate_step(p, st, true);
  if (rc) return rc;
  if ((rc = enter_step(p, st))) return rc;
  if ((rc = flush(p))) return rc;
  return resolve_impl(p, st, nullptr, false);
}

// Launch the gather for every item of a validated, flushed step.  `fused`:
// the step was resolved by the immediately preceding launches, so step-1 rows
// may be copied before the resolve grid finishes (programmatic dependent
// launch; see gather.cu).
static int launch_gathers(dhs_pool* p, const dhs_step* st, bool fused) {
  const dhs_pool_config& c = p->cfg;
  dhs::GatherCommon g{};
  g.tail = (const uint8_t*)c.tail_dev;
  g.opt = (const uint8_t*)c.opt_dev;
  g.hot = (const uint8_t*)c.hot_dev;
  g.map = p->map;
  g.tail_rows = (uint32_t)(p->pairs * c.tail_rows);
  g.opt_rows = (uint32_t)(c.optional_pages * c.page_rows);
  g.hot_rows = (uint32_t)(p->pairs * c.hot_rows);
  g.row_bytes = c.row_bytes;
  g.status = p->status;
  g.T = c.tail_rows;
  g.Pmax = (int32_t)p->pmax;
  g.page_shift = p->page_shift;
  g.early = fused && p->early ? 1 : 0;
  g.trace = p->trace;
  g.loc_ready = p->loc_ready;
  g.fill = p->fill;
  g.fill_words = p->fill_words;
  g.B = c.hot_rows;
  g.later_count = p->later_count;
  g.later_cap = (uint32_t)std::min<int64_t>(p->later_cap, UINT32_MAX);
  g.gen = p->gen;
  g.tpc = p->gather_tpc;
  g.mark_polls = p->mark_polls;
  // the step's resolved items publish their locations; gathers of them (and
  // Reuse items handed the same location vector) may go before the grids end
  const bool lr = fused && p->early && p->fused_resolved && tma_gather(p);
  g.later = lr && use_fresh_list(p) ? p->later : nullptr;
  p->loc_keys.clear();
  if (lr) {
    for (int32_t i = 0; i < st->n_items; ++i) {
      const dhs_item& it = st->items[i];
      if (!(it.flags & DHS_ITEM_GATHER_ONLY) && it.loc_dev)
        p->loc_keys.push_back({it.loc_dev, i, (int64_t)it.req * c.sources + it.src});
    }
    std::sort(p->loc_keys.begin(), p->loc_keys.end());
  }
  // pair whose resolve published `loc`, or -1
  auto loc_pair = [&](const void* loc) -> int64_t {
    auto f = std::upper_bound(p->loc_keys.begin(), p->loc_keys.end(),
                              dhs_pool::LocKey{loc, INT32_MAX, 0});
    if (f == p->loc_keys.begin() || (f - 1)->loc != loc) return -1;
    return (f - 1)->pair;
  };
  // Rows read once: verify queries and Reuse items read their rows again,
  // from L2 when the first read left them there
  g.read_once = 1;
  for (int32_t i = 0; i < st->n_items; ++i)
    if (st->items[i].queries > 1 || (st->items[i].flags & DHS_ITEM_GATHER_ONLY))
      g.read_once = 0;
  p->gitems.clear();
  for (int32_t i = 0; i < st->n_items; ++i) {
    const dhs_item& it = st->items[i];
    const int32_t n = it.queries * it.topk;
    if (n == 0) continue;
    dhs::GatherItem gi{};
    gi.loc = it.loc_dev;
    gi.staging = (uint8_t*)it.staging_dev;
    gi.n = n;
    // a union item's rows are known only once the resolve kernel has ranked
    // them, so it has no early phase
    if (fused && !(it.flags & (DHS_ITEM_GATHER_ONLY | DHS_ITEM_UNION))) {
      const int64_t pair = (int64_t)it.req * c.sources + it.src;
      gi.sel = it.sel_dev;
      gi.pair = (int32_t)pair;
      gi.L = p->ps[pair].L;
      gi.N = p->ps[pair].N;
      gi.L0 = p->l0_of_pair[pair];
      gi.app = p->app_of_pair_rows[pair];
      gi.seq = p->seq_of_pair[pair];
    }
    const int64_t lp = lr ? loc_pair(it.loc_dev) : -1;
    if (lp >= 0) {
      gi.pair = (int32_t)lp;
      gi.seq = p->seq_of_pair[lp];
      gi.flags |= dhs::kGiLocReady;
      // the resolved item itself (not a Reuse item sharing its locations)
      if (it.flags & DHS_ITEM_GATHER_ONLY ? (i < (int32_t)p->staged_item.size() &&
                                             p->staged_item[i])
                                          : p->staged_pair[lp] != 0)
        gi.flags |= dhs::kGiStaged;
    }
    p->gitems.push_back(gi);
  }
  const size_t ng = p->gitems.size();
  const int tile_rows = dhs::gather_tile_rows(p->gather_impl);
  for (size_t b = 0; b < ng; b += dhs::kGatherItemsLarge) {
    const int n = (int)std::min<size_t>(dhs::kGatherItemsLarge, ng - b);
    int64_t tiles = 0, per = -1;
    for (int i = 0; i < n; ++i) {
      dhs::GatherItem& gi = p->gitems[b + i];
      gi.tile0 = (int32_t)tiles;
      const int64_t t = (gi.n + tile_rows - 1) / tile_rows;
      per = i == 0 ? t : (per == t ? per : 0);
      tiles += t;
    }
    if (tiles > INT32_MAX) return DHS_EINVAL;
    g.n_tiles = (int32_t)tiles;
    g.item_tiles = (int32_t)std::max<int64_t>(per, 0);
    // only the first gather launch directly follows the resolve launches
    if (dhs::launch_gather(g, p->gitems.data() + b, n, fused && b == 0, p->gather_impl,
                          p->stream) !=
        cudaSuccess)
      return DHS_ECUDA;
  }
  // the fresh-row list copy runs only when some tile can list a row: an
  // item that waits on published locations and whose fetched rows the host
  // copy does not write itself
  bool listing = false;
  for (const dhs::GatherItem& gi : p->gitems)
    listing |= (gi.flags & dhs::kGiLocReady) && !(gi.flags & dhs::kGiStaged);
  if (g.later && listing &&
      dhs::launch_gather_later(g, 2 * std::max(1, p->sm_count), p->stream) != cudaSuccess)
    return DHS_ECUDA;
  return DHS_OK;
}

// enter_step() for a gather: gathers only read rows, so gathers still
// running on other streams need not be joined.
int enter_gather(dhs_pool* p, const dhs_step* st) {
  p->join_gathers = false;
  const int rc = enter_step(p, st);
  p->join_gathers = true;
  return rc;
}

int dhs_gather(dhs_pool* p, const dhs_step* st) {
  int rc = validate_step(p, st, false);
  if (rc) return rc;
  if ((rc = enter_gather(p, st))) return rc;
  if ((rc = flush(p))) return rc;
  return launch_gathers(p, st, false);
}

int dhs_gather_on(dhs_pool* p, const dhs_step* st, void* stream) {
  if (!p || !stream) return DHS_EINVAL;
  int rc = validate_step(p, st, false);
  if (rc) return rc;
  if ((rc = enter_gather(p, st))) return rc;
  if ((rc = flush(p))) return rc;
  cudaStream_t other = (cudaStream_t)stream;
  cudaEvent_t done = nullptr;
  if (!p->ev_free.empty()) {
    done = p->ev_free.back();
    p->ev_free.pop_back();
  } else if (cudaEventCreateWithFlags(&done, cudaEventDisableTiming) != cudaSuccess) {
    return DHS_ECUDA;
  }
  // after everything the pool's stream holds (resolves, copies, appends)
  if (cudaEventRecord(p->ev_main, p->stream) != cudaSuccess ||
      cudaStreamWaitEvent(other, p->ev_main, 0) != cudaSuccess) {
    p->ev_free.push_back(done);
    return DHS_ECUDA;
  }
  cudaStream_t main = p->stream;
  p->stream = other;
  rc = launch_gathers(p, st, false);
  p->stream = main;
  // joined before the pool's next call that can change rows, even if the
  // launch failed part way
  if (cudaEventRecord(done, other) != cudaSuccess) {
    p->ev_free.push_back(done);
    return DHS_ECUDA;
  }
  p->ev_gathers.push_back(done);
  return rc;
}

int dhs_resolve_gather(dhs_pool* p, const dhs_step* st) {
  int rc = validate_step(p, st, false);
  if (rc) return rc;
  if ((rc = validate_step(p, st, true))) return rc;
  if ((rc = enter(p))) return rc;
  if ((rc = flush(p))) return rc;
  if ((rc = resolve_impl(p, st, nullptr, true))) return rc;
  return launch_gathers(p, st, true);
}

// Validate appends as dhs_append does (distinct admitted pairs, count <= T,
// room left) without launching anything.
static int validate_appends(dhs_pool* p, const dhs_append_item* items, int32_t n_items) {
  if (n_items < 0 || (n_items > 0 && !items)) return DHS_EINVAL;
  const dhs_pool_config& c = p->cfg;
  std::fill(p->seen.begin(), p->seen.end(), 0);
  for (int32_t i = 0; i < n_items; ++i) {
    const dhs_append_item& it = items[i];
    if (it.req < 0 || it.req >= c.max_requests || it.src < 0 || it.src >= c.sources)
      return DHS_EINVAL;
    if (it.count < 0 || it.count > c.tail_rows) return DHS_EINVAL;
    if (it.count > 0 && !it.rows_dev) return DHS_EINVAL;
    const int64_t pair = (int64_t)it.req * c.sources + it.src;
    if (p->seen[pair]) return DHS_EINVAL;
    p->seen[pair] = 1;
    const PairState& s = p->ps[pair];
    if (!s.admitted) return DHS_ESTATE;
    if (s.L + it.count > c.max_rows_per_request) return DHS_EINVAL;
  }
  return DHS_OK;
}

int dhs_decode_step(dhs_pool* p, const dhs_append_item* apps, int32_t n_apps,
                    const dhs_step* st) {
  if (!p) return DHS_EINVAL;
  int rc = validate_appends(p, apps, n_apps);
  if (rc) return rc;
  if ((rc = validate_step(p, st, true))) return rc;
  // fold an append into the resolve kernel only when its pair is resolved
  // in this step; otherwise fall back to a separate append launch
  const dhs_pool_config& c = p->cfg;
  bool foldable = true;
  for (int32_t i = 0; i < n_apps && foldable; ++i) {
    const int64_t pair = (int64_t)apps[i].req * c.sources + apps[i].src;
    foldable = p->seen[pair] != 0 || apps[i].count == 0;  // seen: resolving pairs
  }
  if (!foldable) {
    if ((rc = dhs_append(p, apps, n_apps))) return rc;
    return dhs_resolve_gather(p, st);
  }
  if ((rc = enter(p))) return rc;
  if ((rc = flush(p))) return rc;
  for (int32_t i = 0; i < n_apps; ++i)
    if (apps[i].count > 0)
      p->app_of_pair[(int64_t)apps[i].req * c.sources + apps[i].src] = i;
  rc = resolve_impl(p, st, apps, true);
  for (int32_t i = 0; i < n_apps; ++i)
    p->app_of_pair[(int64_t)apps[i].req * c.sources + apps[i].src] = -1;
  if (rc) return rc;
  return launch_gathers(p, st, true);
}

int dhs_decode_step_host_async(dhs_pool* p, const dhs_copy* in, int32_t n_in,
                               void* in_stream, const dhs_append_item* apps, int32_t n_apps,
                               const dhs_step* st, const dhs_copy* out, int32_t n_out,
                               void* out_stream) {
  if (!p || n_in < 0 || n_out < 0 || (n_in > 0 && !in) || (n_out > 0 && !out))
    return DHS_EINVAL;
  for (int32_t i = 0; i < n_in; ++i)
    if (in[i].bytes && (!in[i].dst || !in[i].src)) return DHS_EINVAL;
  for (int32_t i = 0; i < n_out; ++i)
    if (out[i].bytes && (!out[i].dst || !out[i].src)) return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  cudaStream_t sin = in_stream ? (cudaStream_t)in_stream : p->stream;
  cudaStream_t sout = out_stream ? (cudaStream_t)out_stream : p->stream;
  for (int32_t i = 0; i < n_in; ++i)
    if (in[i].bytes && cudaMemcpyAsync(in[i].dst, in[i].src, in[i].bytes,
                                       cudaMemcpyHostToDevice, sin) != cudaSuccess)
      return DHS_ECUDA;
  if (sin != p->stream && n_in > 0 &&
      (cudaEventRecord(p->ev_in, sin) != cudaSuccess ||
       cudaStreamWaitEvent(p->stream, p->ev_in, 0) != cudaSuccess))
    return DHS_ECUDA;
  if ((rc = dhs_decode_step(p, apps, n_apps, st))) return rc;
  if (sout != p->stream && n_out > 0 &&
      (cudaEventRecord(p->ev_step, p->stream) != cudaSuccess ||
       cudaStreamWaitEvent(sout, p->ev_step, 0) != cudaSuccess))
    return DHS_ECUDA;
  for (int32_t i = 0; i < n_out; ++i)
    if (out[i].bytes && cudaMemcpyAsync(out[i].dst, out[i].src, out[i].bytes,
                                        cudaMemcpyDeviceToHost, sout) != cudaSuccess)
      return DHS_ECUDA;
  return DHS_OK;
}

int dhs_decode_step_host(dhs_pool* p, const dhs_copy* in, int32_t n_in,
                         const dhs_append_item* apps, int32_t n_apps, const dhs_step* st,
                         const dhs_copy* out, int32_t n_out) {
  const int rc = dhs_decode_step_host_async(p, in, n_in, nullptr, apps, n_apps, st, out,
                                            n_out, nullptr);
  if (rc) return rc;
  return cudaStreamSynchronize(p->stream) == cudaSuccess ? DHS_OK : DHS_ECUDA;
}

int dhs_status(dhs_pool* p, uint32_t* flags) {
  if (flags) *flags = 0;
  if (!p) return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, p->status, 4, cudaMemcpyDeviceToHost, p->stream) != cudaSuccess)
    return DHS_ECUDA;
  if (cudaStreamSynchronize(p->stream) != cudaSuccess) return DHS_ECUDA;
  if (v && cudaMemsetAsync(p->status, 0, 4, p->stream) != cudaSuccess) return DHS_ECUDA;
  if (flags) *flags = v;
  if (v & (DHS_STATUS_ERANGE | DHS_STATUS_ELOC)) return DHS_ERANGE;
  if (v & DHS_STATUS_EBUDGET) return DHS_EBUDGET;
  if (v & DHS_STATUS_ETIMEDOUT) return DHS_ETIMEDOUT;
  return DHS_OK;
}

int dhs_read_state(dhs_pool* p, int32_t req, int32_t src, int32_t* tags, uint32_t* stamps,
                   int32_t* page_slot, int64_t* info) {
  if (!p || req < 0 || req >= p->cfg.max_requests || src < 0 || src >= p->cfg.sources)
    return DHS_EINVAL;
  int rc = enter(p);
  if (rc) return rc;
  const int64_t pair = (int64_t)req * p->cfg.sources + src;
  const size_t B = (size_t)p->cfg.hot_rows;
  int32_t st = 0;
  cudaError_t e = cudaSuccess;
  if (tags)
    e = cudaMemcpyAsync(tags, p->tags + pair * B, B * 4, cudaMemcpyDeviceToHost, p->stream);
  if (e == cudaSuccess && stamps)
    e = cudaMemcpyAsync(stamps, p->stamps + pair * B, B * 4, cudaMemcpyDeviceToHost, p->stream);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&st, p->pair_status + pair, 4, cudaMemcpyDeviceToHost, p->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
  if (e != cudaSuccess) return DHS_ECUDA;
  if (page_slot)
    std::memcpy(page_slot, p->map_host.data() + pair * p->pmax, (size_t)p->pmax * 4);
  if (info) {
    const PairState& s = p->ps[pair];
    info[0] = s.N;
    info[1] = s.L;
    info[2] = s.admitted ? 1 : 0;
    info[3] = st;
  }
  return DHS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dhs_resolve_noalloc: dhs_resolve with the miss lists in the library's fixed
// device array instead of the pool's metadata buffer (see include/dhs.h).
extern "C" int dhs_resolve_noalloc(dhs_pool* p, const dhs_step* st) {
  int rc = validate_step(p, st, true);
  if (rc) return rc;
  if (p->pairs > dhs::kNoallocPairs || p->pairs * p->mcap > dhs::kNoallocMissCap)
    return DHS_EINVAL;  // the pool's miss lists do not fit the fixed scratch
  // as dhs_resolve: an outstanding dhs_prefetch is joined only when the step
  // touches its pairs (its miss lists are the pool's, not the fixed array)
  if ((rc = enter_step(p, st))) return rc;
  dhs::NoallocScratch scr{};
  if (dhs::noalloc_scratch(&scr) != cudaSuccess) return DHS_ECUDA;
  if ((rc = flush(p))) return rc;
  return resolve_impl(p, st, nullptr, false, &scr);
}
