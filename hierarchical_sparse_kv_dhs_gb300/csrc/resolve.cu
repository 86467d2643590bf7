// Resolve kernel: a whole CTA per (request, KV source) item of a decode step
// (one CTA per item, or fewer CTAs taking several items each in turn).
//
// "Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
// Hierarchy", How it works / Resolution: a selected row is looked up first
// in the tail ring and the map of GPU-resident optional pages, then among
// the B hot-cache tags (least-recently-used slots give way), and only then
// fetched from its pinned host copy into a hot-cache slot; each row stops at
// the first place that holds it.  Speculative state: the queries of one
// verify block fetch each missing row once between them.
//
// GB300 design.  Everything for one item lives in shared memory:
//   * the union of the Q verify queries is a bitmap over [0, L) (64 rows per
//     word, one optional page per word at 64-row pages), so dedup and
//     ascending order come from the bit positions -- no sort of Q*k ids;
//   * step 1 masks whole words: tail rows by comparison with L-T, optional
//     rows by one page-map read per non-empty word;
//   * step 2 inverts the tag scan: each of the B hot slots tests its tag
//     against the bitmap once (O(B), never more than B probes; tags are
//     unique so the matching slot is the one a linear scan would find);
//   * ranks of unresolved rows come from a block prefix scan of per-word
//     popcounts; misses keep ascending row order by construction;
//   * LRU victims: unprotected slots compacted in slot order, then a stable
//     LSD radix sort on (stamp - min stamp) over only the bits that vary --
//     the first m entries are the m smallest (stamp, slot) keys, which is
//     exactly what evicting one least-recently-used slot at a time for each
//     miss in ascending row order picks;
//   * the misses' (row, slot) pairs go to a global miss list read by the
//     host-copy kernel; locations and counters are written last.
// A window source ("Speculative state": a drafter retains only the rows its
// window covers, stored as a ring) serves only rows [L-T, L): the range check starts
// at the item's `lo`, and every row that passes it is a tail row.
// State (tags, stamps) is written only after the budget check passes, so a
// failing item changes nothing.
#include "dhs_internal.h"

namespace dhs {
namespace {

struct Smem {
  uint64_t* bm;       // [w64cap] selection bitmap, then unresolved-row bitmap
  uint32_t* wpre;     // [w64cap] popcount, then exclusive prefix
  uint32_t* st;       // [B] working stamps
  int32_t* cand_row;  // [qkcap] unresolved rows by rank (ascending)
  uint16_t* slot_of;  // [qkcap] hot slot of each unresolved rank, 0xFFFF = miss
  uint16_t* sort_a;   // [B]
  uint16_t* sort_b;   // [B]
  uint64_t* ubm;      // [w64cap] union bitmap (union staging launches only)
  uint32_t* upre;     // [w64cap] exclusive prefix of its popcounts
  int32_t* sel;       // [selcap] the item's selection, staged (null: read from global)
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline size_t carve(int w64cap, int qkcap, int B, bool uni, int selcap,
                                        Smem* s, unsigned char* base) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align16(off + bytes);
    return base + o;
  };
  unsigned char* p0 = take(sizeof(uint64_t) * (size_t)w64cap);
  unsigned char* p1 = take(sizeof(uint32_t) * (size_t)w64cap);
  unsigned char* p2 = take(sizeof(uint32_t) * (size_t)B);
  unsigned char* p3 = take(sizeof(int32_t) * (size_t)qkcap);
  unsigned char* p4 = take(sizeof(uint16_t) * (size_t)qkcap);
  unsigned char* p5 = take(sizeof(uint16_t) * (size_t)B);
  unsigned char* p6 = take(sizeof(uint16_t) * (size_t)B);
  unsigned char* p7 = uni ? take(sizeof(uint64_t) * (size_t)w64cap) : nullptr;
  unsigned char* p8 = uni ? take(sizeof(uint32_t) * (size_t)w64cap) : nullptr;
  unsigned char* p9 = selcap > 0 ? take(sizeof(int32_t) * (size_t)selcap) : nullptr;
  if (s) {
    s->bm = (uint64_t*)p0;
    s->wpre = (uint32_t*)p1;
    s->st = (uint32_t*)p2;
    s->cand_row = (int32_t*)p3;
    s->slot_of = (uint16_t*)p4;
    s->sort_a = (uint16_t*)p5;
    s->sort_b = (uint16_t*)p6;
    s->ubm = (uint64_t*)p7;
    s->upre = (uint32_t*)p8;
    s->sel = (int32_t*)p9;
  }
  return off;
}

// ---------------------------------------------------------------- block ops
// scratch: 33 uint32 words per independent reduction lane.

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Exclusive prefix of v over the block; *total = block sum.
__device__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  uint32_t inc = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < nw ? scratch[lane] : 0u;
    uint32_t wi = warp_incl_scan(w);
    if (lane < nw) scratch[lane] = wi - w;
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  uint32_t r = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return r;
}

// Exclusive prefix of a 64-bit v over the block (four 16-bit counters
// packed in one word scan at once); *total = block sum.  scratch: 33 words.
__device__ uint64_t block_excl_scan64(uint64_t v, uint64_t* scratch, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  uint64_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint64_t w = lane < nw ? scratch[lane] : 0ull;
    uint64_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) scratch[lane] = wi - w;
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const uint64_t r = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return r;
}

// Sums of four values over the block in one pass.
__device__ void block_sum4(uint32_t v[4], uint32_t* scratch /*[4*33]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[i] += __shfl_xor_sync(0xFFFFFFFFu, v[i], o);
    if (lane == 0) scratch[i * 33 + warp] = v[i];
  }
  __syncthreads();
  if (warp < 4) {
    uint32_t x = lane < nw ? scratch[warp * 33 + lane] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
    if (lane == 0) scratch[warp * 33 + 32] = x;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = scratch[i * 33 + 32];
  __syncthreads();
}

// {sum a, max b, min c, max d} over the block.
__device__ void block_smmm(uint32_t v[4], uint32_t* scratch /*[4*33]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v[0] += __shfl_xor_sync(0xFFFFFFFFu, v[0], o);
    v[1] = max(v[1], __shfl_xor_sync(0xFFFFFFFFu, v[1], o));
    v[2] = min(v[2], __shfl_xor_sync(0xFFFFFFFFu, v[2], o));
    v[3] = max(v[3], __shfl_xor_sync(0xFFFFFFFFu, v[3], o));
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) scratch[i * 33 + warp] = v[i];
  }
  __syncthreads();
  if (warp < 4) {
    const uint32_t ident = warp == 2 ? 0xFFFFFFFFu : 0u;
    uint32_t x = lane < nw ? scratch[warp * 33 + lane] : ident;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, o);
      x = warp == 0 ? x + y : (warp == 2 ? min(x, y) : max(x, y));
    }
    if (lane == 0) scratch[warp * 33 + 32] = x;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = scratch[i * 33 + 32];
  __syncthreads();
}

// In-place exclusive scan of a[0, n); returns the total.
__device__ uint32_t block_scan_array(uint32_t* a, int n, uint32_t* scratch) {
  const int per = (n + (int)blockDim.x - 1) / (int)blockDim.x;
  const int b = (int)threadIdx.x * per;
  const int e = min(n, b + per);
  uint32_t s = 0;
  for (int i = b; i < e; ++i) s += a[i];
  uint32_t total;
  uint32_t pre = block_excl_scan(s, scratch, &total);
  for (int i = b; i < e; ++i) {
    uint32_t t = a[i];
    a[i] = pre;
    pre += t;
  }
  __syncthreads();
  return total;
}

// OR a 64-bit mask into a shared bitmap word as two 32-bit atomics (only
// the halves that have bits): 32-bit shared-memory atomics are native.
__device__ __forceinline__ void or_word(uint64_t* word, uint64_t bits) {
  uint32_t* w = reinterpret_cast<uint32_t*>(word);
  const uint32_t lo = (uint32_t)bits, hi = (uint32_t)(bits >> 32);
  if (lo) atomicOr(w, lo);
  if (hi) atomicOr(w + 1, hi);
}

// ---------------------------------------------------------------- masks

// Rows of word w (rows 64w .. 64w+63) that lie in the tail [t0, ...).
__device__ __forceinline__ uint64_t tail_mask(int w, int64_t t0) {
  const int64_t lo = (int64_t)w << 6;
  if (lo >= t0) return ~0ull;
  if (lo + 63 < t0) return 0ull;
  return ~0ull << (int)(t0 - lo);
}

// Rows of word w in complete imported pages whose optional slot is ready.
__device__ __forceinline__ uint64_t opt_mask(int w, int64_t N, const int32_t* map,
                                             int ps) {
  const int64_t lo = (int64_t)w << 6;
  if (ps >= 6) {
    const int64_t page = lo >> ps;
    return (((page + 1) << ps) <= N && map[page] >= 0) ? ~0ull : 0ull;
  }
  const int rows = 1 << ps;
  const uint64_t one = (rows == 64) ? ~0ull : ((1ull << rows) - 1ull);
  uint64_t m = 0;
  for (int i = 0; i < (64 >> ps); ++i) {
    const int64_t page = (lo >> ps) + i;
    if (((page + 1) << ps) <= N && map[page] >= 0) m |= one << (i * rows);
  }
  return m;
}

// Rank of a row among the set bits of a bitmap over [0, L), given the
// exclusive prefix of the words' bit counts.
__device__ __forceinline__ uint32_t union_rank(const uint64_t* bm, const uint32_t* pre,
                                               int32_t row) {
  const uint64_t bit = 1ull << (row & 63);
  return pre[row >> 6] + (uint32_t)__popcll(bm[row >> 6] & (bit - 1ull));
}

// Position of the k-th set bit (from 0) of a word holding more than k bits,
// by halving: count the low half's bits, step into the half that holds it.
__device__ __forceinline__ int nth_set_bit(uint64_t m, uint32_t k) {
  int pos = 0;
#pragma unroll
  for (int w = 32; w >= 1; w >>= 1) {
    const uint64_t low = m & ((1ull << w) - 1ull);
    const uint32_t c = (uint32_t)__popcll(low);
    if (k >= c) {
      k -= c;
      pos += w;
      m >>= w;
    } else {
      m = low;
    }
  }
  return pos;
}

// The row of union rank u (u below the union's size): the last word whose
// prefix is at most u holds it (empty words share the next word's prefix).
__device__ __forceinline__ int32_t union_row(const uint64_t* bm, const uint32_t* pre, int W,
                                             uint32_t u) {
  int lo = 0, hi = W - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return (lo << 6) + nth_set_bit(bm[lo], u - pre[lo]);
}

// Publish that an item's locations (and the decode rows it appended) are
// written (thread 0 only, after a block barrier).
__device__ __forceinline__ void publish_loc(const ResolveCommon& c, int pair) {
  if (!c.loc_ready) return;
  __threadfence();
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(c.loc_ready + pair),
               "r"(c.seq & kSeqMask) : "memory");
}

// Publish that an item's miss count and miss lists are written, and its
// staging entries too unless `pending` (thread 0 only, after a block
// barrier): its host copy may start.  A pending mark is followed by a second
// one without the bit once the entries are written.  An item without misses
// says so in the mark itself; the copy then reads nothing the item wrote, so
// the mark needs no fence (a fence waits for the block's earlier writes,
// microseconds while the gather fills the memory system).
__device__ __forceinline__ void publish_copy(const ResolveCommon& c, int pair, bool none,
                                             bool pending = false) {
  if (!c.copy_ready) return;
  if (!none) __threadfence();
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(c.copy_ready + pair),
               "r"((c.seq & kSeqMask) | (none ? kMarkNoMiss : 0u) |
                   (pending ? kMarkEntriesPending : 0u)) : "memory");
}

// Write the failure result of one item: no state change, zero counters.
// Step 1 of "Resolution" reads no state that resolution changes, so the
// entries it resolves keep their locations (the tail, or a ready page of the
// optional map) and every other entry gets none; the fused gather copies
// step-1 rows without waiting for the outcome.  A union item gets an empty
// list.
__device__ void fail_item(const ResolveCommon& c, const ResolveItem& it, int32_t code,
                          uint32_t flag) {
  if (it.index) {  // union staging: an empty union list
    for (int e = threadIdx.x; e < it.n; e += blockDim.x) {
      it.loc[e] = kEndLoc;
      it.index[e] = -1;
    }
  } else {
    const int64_t L = it.L, N = it.N, T = c.T;
    const int ps = c.page_shift;
    const int32_t* map = c.map + (size_t)it.pair * c.Pmax;
    for (int e = threadIdx.x; e < it.n; e += blockDim.x) {
      const int32_t row = it.sel[e];
      uint32_t l = kNoLoc;
      if (row >= 0 && (int64_t)row < L) {
        const int64_t page = (int64_t)row >> ps;
        if ((int64_t)row >= L - T) {
          l = (kTierTail << 30) | (uint32_t)((int64_t)it.pair * T + (int64_t)row % T);
        } else if (((page + 1) << ps) <= N && map[page] >= 0) {
          l = (kTierOpt << 30) |
              (uint32_t)(((int64_t)map[page] << ps) + (row & ((1 << ps) - 1)));
        }
      }
      it.loc[e] = l;
    }
  }
  if (threadIdx.x < 8 && it.counters) it.counters[threadIdx.x] = 0u;
  __syncthreads();
  if (threadIdx.x == 0) {
    c.miss_count[it.pair] = 0u;  // before the marks: the host copy reads it then
    c.copy_cursor[it.pair] = 0u;
    c.pair_status[it.pair] = code;
    publish_copy(c, it.pair, true);
    publish_loc(c, it.pair);
    atomicOr(c.status, flag);
    trace_mark(c.trace, kTraceResolve, true);
  }
}

// ---------------------------------------------------------------- kernel

template <int MAXI>
struct ResolveParams {
  ResolveCommon c;
  ResolveItem items[MAXI];
};
// kernel parameter space holds at most 32764 bytes
static_assert(sizeof(ResolveParams<kResolveItemsLarge>) <= 32764, "resolve item table too large");

// Resolve launch item `item` with the whole CTA (every return is taken by
// all its threads alike).
template <int MAXI>
__device__ __forceinline__ void resolve_one(const ResolveParams<MAXI>& P, const int item,
                                            unsigned char* smem_raw, uint32_t* scratch,
                                            uint64_t* scratch64, int& s_bad) {
  const ResolveCommon& c = P.c;
  const ResolveItem& it = P.items[item];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int B = c.B;
  const int64_t T = c.T;
  const int64_t L = it.L, N = it.N;
  const int64_t t0 = L - T;
  const int n = it.n;
  const int W = (int)((L + 63) >> 6);
  const uint32_t step = c.step;
  const int pair = it.pair;
  int32_t* tags = c.tags + (size_t)pair * B;
  uint32_t* stamps = c.stamps + (size_t)pair * B;
  const int32_t* map = c.map + (size_t)pair * c.Pmax;

  // this step's fill marks start empty; the next fused step's fresh-row
  // list starts empty (nothing reads either before this launch completes
  // or, for the fill marks, before this item publishes its locations)
  uint32_t* fill = c.fill ? c.fill + (size_t)pair * c.fill_words : nullptr;
  if (fill)
    for (int j = tid; j < c.fill_words; j += nt) fill[j] = 0u;
  if (c.later_count && item == 0 && tid == 0) c.later_count[(c.gen & 1u) ^ 1u] = 0u;

  Smem s;
  carve(c.w64cap, c.qkcap, B, c.uni != 0, c.selcap, &s, smem_raw);
  // The selection is read by several passes.  A large one (at least eight
  // entries per thread: verify blocks) is staged in shared memory once, with
  // coalesced loads, eight in flight per thread, when the launch's plan has
  // room; a small one is read from global memory by each pass (staging it
  // costs one more round of load latency than it saves).
  const bool staged = s.sel != nullptr && it.n <= c.selcap && it.n >= 8 * nt;
  if (staged) {
    for (int e0 = tid; e0 < it.n; e0 += 8 * nt) {
      int32_t v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = e0 + u * nt < it.n ? it.sel[e0 + u * nt] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * nt < it.n) s.sel[e0 + u * nt] = v[u];
    }
    __syncthreads();
  }
  const int32_t* sel = staged ? s.sel : it.sel;
  // f(entry, row) over every entry of the selection, each thread issuing the
  // loads of four entries before using them
  auto for_entries = [&](auto&& f) {
    for (int e0 = tid; e0 < it.n; e0 += 4 * nt) {
      int32_t r4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * nt;
        r4[u] = e < it.n ? sel[e] : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * nt;
        if (e < it.n) f(e, r4[u]);
      }
    }
  };
  const bool uni = it.index != nullptr;  // union staging (launch has c.uni)

  // ---- decode rows appended by this launch (dhs_decode_step): row L0+j to
  // tail slot (L0+j) mod T and through to the pinned host copy.  Nothing
  // below reads them; the gather reads them only after this grid completes.
  if (it.app_count) {
    const int rb = c.row_bytes, cpr = rb >> 4;
    const int total = it.app_count * cpr;
    for (int ch = tid; ch < total; ch += nt) {
      const int j = ch / cpr, p = ch - j * cpr;
      const int64_t row = it.app_L0 + j;
      const uint4 v = *reinterpret_cast<const uint4*>(it.app_rows + (size_t)j * rb + p * 16);
      *reinterpret_cast<uint4*>(c.tail + ((size_t)pair * T + (size_t)(row % T)) * rb +
                                p * 16) = v;
      if (it.app_host) *reinterpret_cast<uint4*>(it.app_host + (size_t)row * rb + p * 16) = v;
    }
  }

  // ---- union of the verify block as a bitmap; range check
  for (int w = tid; w < W; w += nt) s.bm[w] = 0ull;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  // Each thread takes a run of consecutive entries (at least four: one run
  // per thread when the selection is large), ORs the bits that fall in one
  // 64-row word into a register and updates shared memory once per word it
  // touches.  Selections cluster (a recency window, sorted top-k lists; a
  // verify block repeats the same window in every query), so this is about
  // one atomic per run instead of one per entry, many on the same word.
  const int run = max(4, (((n + nt - 1) / nt) + 3) & ~3);
  for (int b = tid * run; b < n; b += nt * run) {
    uint64_t acc = 0ull;
    int cur = -1;
    const int end = min(n, b + run);
    for (int j0 = b; j0 < end; j0 += 4) {
      int32_t r4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) r4[u] = j0 + u < end ? sel[j0 + u] : 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (j0 + u >= end) break;
        const int32_t row = r4[u];
        if ((int64_t)row < it.lo || (int64_t)row >= L) {
          s_bad = 1;
          continue;
        }
        const int w = row >> 6;
        if (w != cur) {
          if (cur >= 0) or_word(&s.bm[cur], acc);
          cur = w;
          acc = 0ull;
        }
        acc |= 1ull << (row & 63);
      }
    }
    if (cur >= 0) or_word(&s.bm[cur], acc);
  }
  __syncthreads();
  if (s_bad) {
    fail_item(c, it, kErrRange, kStatusErange);
    return;
  }

  // ---- step 1: tail and ready optional map, word by word
  uint32_t cnt[4] = {0u, 0u, 0u, 0u};  // unique, tail, opt, unresolved
  for (int w = tid; w < W; w += nt) {
    const uint64_t bits = s.bm[w];
    if (uni) {
      s.ubm[w] = bits;
      s.upre[w] = (uint32_t)__popcll(bits);
    }
    uint64_t cand = 0ull;
    if (bits) {
      const uint64_t tm = bits & tail_mask(w, t0);
      const uint64_t rest = bits & ~tm;
      const uint64_t om = rest ? (rest & opt_mask(w, N, map, c.page_shift)) : 0ull;
      cand = rest & ~om;
      cnt[0] += __popcll(bits);
      cnt[1] += __popcll(tm);
      cnt[2] += __popcll(om);
      cnt[3] += __popcll(cand);
    }
    s.bm[w] = cand;
    s.wpre[w] = (uint32_t)__popcll(cand);
  }
  block_sum4(cnt, scratch);
  const uint32_t n_unique = cnt[0], n_tail = cnt[1], n_opt = cnt[2];
  const uint32_t C = cnt[3];  // rows left for the hot cache (block-uniform)
  if (uni) block_scan_array(s.upre, W, scratch);  // union ranks

  // More rows left for the hot cache than it has slots: whatever the scan
  // finds, the misses (C - hits) outnumber the unprotected slots (at most
  // B - hits), so the item fails the budget now -- and the candidate arrays,
  // sized for B rows, are never filled past their end.
  if (C > (uint32_t)B) {
    fail_item(c, it, kErrBudget, kStatusEbudget);
    return;
  }
  uint32_t hits = 0u, m_miss = 0u, scan_max = 0u, evicted = 0u;
  if (C) {
    block_scan_array(s.wpre, W, scratch);  // candidate ranks
    for (int j = tid; j < B; j += nt) s.st[j] = stamps[j];
    // rank -> row for the unresolved rows (ascending)
    for (int w = tid; w < W; w += nt) {
      uint64_t m = s.bm[w];
      uint32_t r = s.wpre[w];
      while (m) {
        const int b = __ffsll((long long)m) - 1;
        m &= m - 1;
        s.cand_row[r] = (w << 6) + b;
        s.slot_of[r] = 0xFFFFu;
        ++r;
      }
    }
    __syncthreads();

    // ---- step 2: every hot slot tests its tag once (B probes in total)
    uint32_t hv0 = 0u, hv1 = 0u;  // hits, max probes
    for (int j = tid; j < B; j += nt) {
      const int32_t t = tags[j];
      if (t >= 0 && (int64_t)t < L) {
        const uint64_t m = s.bm[t >> 6];
        const uint64_t bit = 1ull << (t & 63);
        if (m & bit) {
          const uint32_t r = s.wpre[t >> 6] + (uint32_t)__popcll(m & (bit - 1ull));
          s.slot_of[r] = (uint16_t)j;
          s.st[j] = step;
          hv0 += 1u;
          hv1 = max(hv1, (uint32_t)(j + 1));
        }
      }
    }
    __syncthreads();
    // unprotected slots and their stamp range
    uint32_t un = 0u, umin = 0xFFFFFFFFu, umax = 0u;
    for (int j = tid; j < B; j += nt) {
      const uint32_t x = s.st[j];
      if (x != step) {
        un += 1u;
        umin = min(umin, x);
        umax = max(umax, x);
      }
    }
    uint32_t red[4] = {hv0, hv1, umin, umax};  // {sum, max, min, max}
    block_smmm(red, scratch);
    uint32_t cnt2[4] = {un, 0u, 0u, 0u};
    block_sum4(cnt2, scratch);
    hits = red[0];
    m_miss = C - hits;
    const uint32_t unprot = cnt2[0];
    scan_max = m_miss ? (uint32_t)B : red[1];

    if (m_miss > unprot) {  // more missing rows than victims: change nothing
      fail_item(c, it, kErrBudget, kStatusEbudget);
      return;
    }

    // ---- step 3 victims: the m smallest (stamp, slot) among unprotected slots
    if (m_miss) {
      {  // stable compaction of unprotected slots, ascending slot order
        const int per = (B + nt - 1) / nt;
        const int b = tid * per, e = min(B, b + per);
        uint32_t u = 0;
        for (int j = b; j < e; ++j) u += s.st[j] != step;
        uint32_t tot;
        uint32_t pos = block_excl_scan(u, scratch, &tot);
        for (int j = b; j < e; ++j)
          if (s.st[j] != step) s.sort_a[pos++] = (uint16_t)j;
        __syncthreads();
      }
      const uint32_t kmin = red[2];
      const uint32_t span = red[3] - kmin;
      const int nbits = span ? 32 - __clz(span) : 0;
      uint16_t* src = s.sort_a;
      uint16_t* dst = s.sort_b;
      const int U = (int)unprot;
      const int per = (U + nt - 1) / nt;
      const int b = tid * per, e = min(U, b + per);
      // stable LSD radix sort, two bits per pass: each thread counts the four
      // digits of its contiguous range in 16-bit fields of one word (U <=
      // 16384 fits), one block scan gives every thread its place in each
      // digit's bucket, and each range is written out in order
      for (int sh = 0; sh < nbits; sh += 2) {
        uint64_t cnt = 0ull;
        for (int i = b; i < e; ++i)
          cnt += 1ull << (16u * (((s.st[src[i]] - kmin) >> sh) & 3u));
        uint64_t tot;
        const uint64_t pre = block_excl_scan64(cnt, scratch64, &tot);
        // bucket d starts after every smaller digit's total; this thread's
        // place in it is its prefix field (positions packed like the counts)
        const uint64_t t0 = tot & 0xFFFFull, t1 = (tot >> 16) & 0xFFFFull,
                       t2 = (tot >> 32) & 0xFFFFull;
        uint64_t pos = pre + ((t0 << 16) | ((t0 + t1) << 32) | ((t0 + t1 + t2) << 48));
        for (int i = b; i < e; ++i) {
          const uint16_t v = src[i];
          const uint32_t sh16 = 16u * (((s.st[v] - kmin) >> sh) & 3u);
          dst[(uint32_t)(pos >> sh16) & 0xFFFFu] = v;
          pos += 1ull << sh16;
        }
        __syncthreads();
        uint16_t* t = src;
        src = dst;
        dst = t;
      }
      // i-th missing row (ascending) -> i-th victim
      {
        const int perc = ((int)C + nt - 1) / nt;
        const int cb = tid * perc, ce = min((int)C, cb + perc);
        uint32_t mm = 0;
        for (int i = cb; i < ce; ++i) mm += s.slot_of[i] == 0xFFFFu;
        uint32_t mtot;
        uint32_t mr = block_excl_scan(mm, scratch, &mtot);
        int32_t* mrows = c.miss_rows + (size_t)pair * c.Mcap;
        int32_t* mslots = c.miss_slots + (size_t)pair * c.Mcap;
        for (int i = cb; i < ce; ++i) {
          if (s.slot_of[i] != 0xFFFFu) continue;
          const int v = src[mr];
          const int32_t row = s.cand_row[i];
          evicted += tags[v] != -1;
          if (fill) atomicOr(&fill[v >> 5], 1u << (v & 31));
          tags[v] = row;
          s.st[v] = step;
          s.slot_of[i] = (uint16_t)v;
          s.cand_row[i] = ~(int32_t)mr;  // from here on: miss index of candidate i
          mrows[mr] = row;
          mslots[mr] = v;
          ++mr;
        }
      }
      __syncthreads();
    }

    // ---- commit stamps of every slot hit or filled in this step
    for (int j = tid; j < B; j += nt)
      if (s.st[j] == step) stamps[j] = step;
  }

  // A per-query item's staging entries take two passes over its selection
  // (about 11 us of a C64 CTA's 38): its miss lists go out first, marked
  // with the entries pending, so that its host copy can read the rows and
  // fill their hot slots meanwhile, and writes staging once the second mark
  // is out.
  const bool entries_later = it.stage && m_miss && !uni;
  if (entries_later) {
    __syncthreads();  // every thread's miss-list writes are done
    if (tid == 0) {
      c.miss_count[pair] = m_miss;
      c.copy_cursor[pair] = 0u;  // the copy's blocks claim rows from here
      publish_copy(c, pair, false, true);
    }
  }

  // ---- staging entries of each miss (the host copy writes them): entries
  // grouped by miss index, CSR in miss_off / miss_ent.  After the stamp
  // commit the working stamps serve as per-miss counters, then cursors.
  if (it.stage && m_miss && uni) {
    // one staging row per distinct row: a miss's only staging entry is its
    // row's rank in the union, so miss i takes entry i
    int32_t* off = c.miss_off + (size_t)pair * (c.Mcap + 1);
    int32_t* ent = c.miss_ent + (size_t)pair * c.ent_cap;
    const int32_t* mrows = c.miss_rows + (size_t)pair * c.Mcap;
    __syncthreads();
    for (uint32_t j = tid; j < m_miss; j += nt) {
      const int32_t row = mrows[j];
      off[j] = (int32_t)j;
      ent[j] = (int32_t)union_rank(s.ubm, s.upre, row);
    }
    if (tid == 0) off[m_miss] = (int32_t)m_miss;
  } else if (it.stage && m_miss) {
    int32_t* off = c.miss_off + (size_t)pair * (c.Mcap + 1);
    int32_t* ent = c.miss_ent + (size_t)pair * c.ent_cap;
    // miss index of the entry's row, or -1 when the row is not a miss
    auto miss_of = [&](int32_t row) -> int32_t {
      if ((int64_t)row >= t0) return -1;
      const uint64_t m = s.bm[row >> 6];
      const uint64_t bit = 1ull << (row & 63);
      if (!(m & bit)) return -1;
      const int32_t v = s.cand_row[s.wpre[row >> 6] + (uint32_t)__popcll(m & (bit - 1ull))];
      return v < 0 ? ~v : -1;
    };
    __syncthreads();
    for (uint32_t j = tid; j < m_miss; j += nt) s.st[j] = 0u;
    __syncthreads();
    for_entries([&](int, int32_t row) {
      const int32_t mi = miss_of(row);
      if (mi >= 0) atomicAdd(&s.st[mi], 1u);
    });
    __syncthreads();
    const uint32_t total = block_scan_array(s.st, (int)m_miss, scratch);
    for (uint32_t j = tid; j < m_miss; j += nt) off[j] = (int32_t)s.st[j];
    if (tid == 0) off[m_miss] = (int32_t)total;
    __syncthreads();
    for_entries([&](int e, int32_t row) {
      const int32_t mi = miss_of(row);
      if (mi >= 0) ent[atomicAdd(&s.st[mi], 1u)] = e;
    });
  }
  __syncthreads();
  if (tid == 0) {
    // the miss count, miss lists and staging entries are written: the host
    // copy of this item may start (or write staging) while its locations
    // are being written
    if (!entries_later) {
      c.miss_count[pair] = m_miss;
      c.copy_cursor[pair] = 0u;  // the copy's blocks claim rows from here
    }
    publish_copy(c, pair, m_miss == 0);
  }

  // ---- location vector
  const int ps = c.page_shift;
  const int64_t pmask = ((int64_t)1 << ps) - 1;
  auto loc_of = [&](int32_t row) -> uint32_t {
    if ((int64_t)row >= t0)
      return (kTierTail << 30) | (uint32_t)((int64_t)pair * T + (int64_t)row % T);
    const uint64_t m = s.bm[row >> 6];  // rows that went to the hot cache
    const uint64_t bit = 1ull << (row & 63);
    if (m & bit) {
      const uint32_t r = s.wpre[row >> 6] + (uint32_t)__popcll(m & (bit - 1ull));
      return (kTierHot << 30) | (uint32_t)((int64_t)pair * B + s.slot_of[r]);
    }
    const int32_t slot = map[row >> ps];
    return (kTierOpt << 30) | (uint32_t)(((int64_t)slot << ps) + (row & pmask));
  };
  if (!uni) {
    // four locations computed (their page-map loads in flight together)
    // before they are stored
    for (int e0 = tid; e0 < n; e0 += 4 * nt) {
      int32_t r4[4];
      uint32_t l4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = e0 + u * nt;
        r4[u] = e < n ? sel[e] : 0;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) l4[u] = e0 + u * nt < n ? loc_of(r4[u]) : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (e0 + u * nt < n) it.loc[e0 + u * nt] = l4[u];
    }
  } else {
    // union staging: each entry's rank among the distinct rows, the distinct
    // rows' locations in ascending row order, then the end marker
    for (int e = tid; e < n; e += nt) it.index[e] = (int32_t)union_rank(s.ubm, s.upre, sel[e]);
    // rank u's row: the word whose rank range holds u (binary search of the
    // word prefix), then the matching set bit; four ranks a thread in flight,
    // stores coalesced
    for (int u0 = tid; u0 < (int)n_unique; u0 += 4 * nt) {
      int32_t r4[4];
      uint32_t l4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int u = u0 + q * nt;
        r4[q] = u < (int)n_unique ? union_row(s.ubm, s.upre, W, (uint32_t)u) : 0;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) l4[q] = u0 + q * nt < (int)n_unique ? loc_of(r4[q]) : 0u;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (u0 + q * nt < (int)n_unique) it.loc[u0 + q * nt] = l4[q];
    }
    for (int u = (int)n_unique + tid; u < n; u += nt) it.loc[u] = kEndLoc;
  }
  __syncthreads();
  if (tid == 0) {
    c.pair_status[pair] = 0;
    // everything the gather reads of this item -- locations, fill marks,
    // appended rows -- is written before the mark.  Only tiles with rows that
    // step 1 leaves open (hot-cache rows, a union list, a gather-only item
    // reading this vector) wait for it; without such rows nothing does, and
    // the mark and its fence are left out.
    if (C != 0u || uni || it.loc_shared) publish_loc(c, pair);
  }

  if (m_miss) {
    uint32_t ev[4] = {evicted, 0u, 0u, 0u};
    block_sum4(ev, scratch);
    evicted = ev[0];
  }
  if (tid == 0) {
    if (it.counters) {
      it.counters[0] = (uint32_t)n;
      it.counters[1] = n_unique;
      it.counters[2] = n_tail;
      it.counters[3] = n_opt;
      it.counters[4] = hits;
      it.counters[5] = m_miss;
      it.counters[6] = scan_max;
      it.counters[7] = evicted;
    }
    trace_mark(c.trace, kTraceResolve, true);
  }
}

// CTA b resolves items b, b + gridDim, ... one after the other (one item per
// CTA unless the launch asks for fewer CTAs than items).
template <int MAXI, int THREADS, int MINB>
__global__ void __launch_bounds__(THREADS, MINB)
    resolve_kernel(const __grid_constant__ ResolveParams<MAXI> P) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint32_t scratch[4 * 33];
  __shared__ uint64_t scratch64[33];
  __shared__ int s_bad;

  // Dependent launches (the host copy, then the gather) may start now: they
  // wait for this grid's completion, or for an item's marks, before reading
  // anything it writes.
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) trace_mark(P.c.trace, kTraceResolve, false);
  for (int item = blockIdx.x; item < P.c.n_items; item += gridDim.x) {
    resolve_one(P, item, smem_raw, scratch, scratch64, s_bad);
    __syncthreads();  // the next item reuses the shared-memory plan
  }
}

template <int MAXI, int THREADS, int MINB>
cudaError_t launch_t(const ResolveCommon& c, const ResolveItem* items, int n, int ctas,
                     size_t smem, cudaStream_t stream) {
  ResolveParams<MAXI> P;
  P.c = c;
  P.c.n_items = n;
  for (int i = 0; i < n; ++i) P.items[i] = items[i];
  const int grid = ctas > 0 && ctas < n ? ctas : n;
  resolve_kernel<MAXI, THREADS, MINB><<<grid, THREADS, smem, stream>>>(P);
  return cudaGetLastError();
}

// the three instances: small launches, large launches, large launches two per SM
#define DHS_RESOLVE_SMALL kResolveItemsSmall, resolve_threads(kResolveItemsSmall), 1
#define DHS_RESOLVE_LARGE kResolveItemsLarge, resolve_threads(kResolveItemsLarge), 1
#define DHS_RESOLVE_PAIRED kResolveItemsLarge, kResolvePairThreads, 2

}  // namespace

size_t resolve_smem_bytes(int w64cap, int qkcap, int B, bool uni, int selcap) {
  return carve(w64cap, qkcap, B, uni, selcap, nullptr, nullptr);
}

cudaError_t resolve_set_smem_limit(size_t bytes) {
  // The attribute is per function and device; only ever raise it, so a
  // smaller pool created later never breaks a larger one.
  static int device_limit[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    if ((int)bytes <= device_limit[dev]) return cudaSuccess;
    device_limit[dev] = (int)bytes;
  }
  for (const void* k : {(const void*)resolve_kernel<DHS_RESOLVE_SMALL>,
                        (const void*)resolve_kernel<DHS_RESOLVE_LARGE>,
                        (const void*)resolve_kernel<DHS_RESOLVE_PAIRED>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t resolve_set_carveout() {
  for (const void* k : {(const void*)resolve_kernel<DHS_RESOLVE_SMALL>,
                        (const void*)resolve_kernel<DHS_RESOLVE_LARGE>,
                        (const void*)resolve_kernel<DHS_RESOLVE_PAIRED>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_resolve(const ResolveCommon& c, const ResolveItem* items,
                           int n_items, int ctas, size_t smem, bool paired,
                           cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (n_items <= kResolveItemsSmall)
    return launch_t<DHS_RESOLVE_SMALL>(c, items, n_items, ctas, smem, stream);
  if (paired) return launch_t<DHS_RESOLVE_PAIRED>(c, items, n_items, ctas, smem, stream);
  return launch_t<DHS_RESOLVE_LARGE>(c, items, n_items, ctas, smem, stream);
}

}  // namespace dhs
