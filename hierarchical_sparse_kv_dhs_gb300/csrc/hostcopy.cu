// Host-copy kernel: step 3 of resolution, the fetch of a row that neither
// the tail, the resident optional pages nor the hot cache holds, from its
// pinned host copy into a hot-cache slot ("Adaptive DHiSparse", How it
// works / Resolution).
//
// Reads the missing rows straight out of mapped pinned host memory over
// NVLink-C2C into their victim hot-cache slots.  The pages size the copy
// kernel's grid between 4 and 32 blocks by batch size; on GB300 fewer than
// about 16 blocks leave the host link idle, so the grid is at least the
// upper end, 32 blocks of 512 threads, whatever the batch (a claiming launch
// of more items than SMs runs the same warps as 64 blocks of 256, leaving
// room beside each for gather CTAs).  The pool grows it further when
// the items' pinned regions are large (each block's share kept within about
// 1 GiB, so that the translations of its rows stay cached near its SM).
// Within 16 GiB of pinned rows the blocks claim rows through per-item
// cursors and take each other's leftovers.  Past that each block keeps to
// its own items and reserves its SM's shared memory, so that no gather CTA
// lands beside it; the copy then launches after the resolve grid, so that
// block b lands on the same SM every step, unless every copy block finds an
// SM that the resolve grid leaves free.  Each warp keeps up to four
// 1152-byte rows in flight (12 x 16-byte loads per lane) so the link sees
// enough outstanding requests to cover its latency.
#include <algorithm>

#include "dhs_internal.h"

namespace dhs {
namespace {

template <int MAXI>
struct CopyParams {
  CopyCommon c;
  CopyItem items[MAXI];
};
// kernel parameter space holds at most 32764 bytes
static_assert(sizeof(CopyParams<kCopyItemsMax>) <= 32764, "copy item table too large");

__device__ __forceinline__ uint4 ld_sys(const uint8_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

constexpr int kRowsPerWarp = 4;
constexpr int kChunksPerLane = 3;  // rows up to 96 x 16 = 1536 bytes

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Copy misses [r0, r1) (at most kRowsPerWarp) of one item: one warp of the
// claiming copy.  Each row goes to its victim hot slot and, for items whose
// host copy stages, to its staging entries (miss_off / miss_ent) in the
// item's staging and in that of the gather-only items sharing its
// locations.  wait_entries() returns once those entries are written; the
// rows' host reads and hot-slot writes go ahead of it.
template <bool kSmallRow, int MAXI, typename WaitEntries>
__device__ __forceinline__ void copy_rows(const CopyParams<MAXI>& P, const CopyItem& it,
                                          uint32_t r0, uint32_t r1, int lane,
                                          WaitEntries&& wait_entries) {
  const CopyCommon& c = P.c;
  const int rb = c.row_bytes, cpr = rb >> 4;
  const size_t base = (size_t)it.pair * c.Mcap;
  const uint8_t* src[kRowsPerWarp];
  uint8_t* dst[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const uint32_t i = r0 + r;
    src[r] = nullptr;
    dst[r] = nullptr;
    if (i < r1) {
      src[r] = it.host + (size_t)c.miss_rows[base + i] * rb;
      dst[r] = c.hot + ((size_t)it.pair * c.B + c.miss_slots[base + i]) * rb;
    }
  }
  const int32_t* mo = c.miss_off + (size_t)it.pair * (c.Mcap + 1);
  const int32_t* ents = c.miss_ent + (size_t)it.pair * c.ent_cap;
  if (kSmallRow) {
    uint4 v[kRowsPerWarp][kChunksPerLane];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int q = 0; q < kChunksPerLane; ++q) {
        const int ch = lane + 32 * q;
        if (src[r] && ch < cpr) v[r][q] = ld_sys(src[r] + ch * 16);
      }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int q = 0; q < kChunksPerLane; ++q) {
        const int ch = lane + 32 * q;
        if (dst[r] && ch < cpr) *reinterpret_cast<uint4*>(dst[r] + ch * 16) = v[r][q];
      }
    if (!it.staging) return;
    wait_entries();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (!src[r]) continue;
      const uint32_t i = r0 + r;
      for (int k = mo[i]; k < mo[i + 1]; ++k) {
        const size_t eo = (size_t)ents[k] * rb;
        for (int j = -1; j < it.nshare; ++j) {
          uint8_t* to = (j < 0 ? it.staging : it.share[j]) + eo;
#pragma unroll
          for (int q = 0; q < kChunksPerLane; ++q) {
            const int ch = lane + 32 * q;
            if (ch < cpr) *reinterpret_cast<uint4*>(to + ch * 16) = v[r][q];
          }
        }
      }
    }
  } else {
    if (it.staging) wait_entries();
    for (int r = 0; r < kRowsPerWarp; ++r) {
      if (!src[r]) continue;
      const uint32_t i = r0 + r;
      const int e0 = it.staging ? mo[i] : 0, e1 = it.staging ? mo[i + 1] : 0;
      for (int ch = lane; ch < cpr; ch += 32) {
        const uint4 v = ld_sys(src[r] + ch * 16);
        *reinterpret_cast<uint4*>(dst[r] + ch * 16) = v;
        for (int k = e0; k < e1; ++k) {
          const size_t eo = (size_t)ents[k] * rb + ch * 16;
          *reinterpret_cast<uint4*>(it.staging + eo) = v;
          for (int j = 0; j < it.nshare; ++j) *reinterpret_cast<uint4*>(it.share[j] + eo) = v;
        }
      }
    }
  }
}

// Copy the miss rows of the launch's items.  An item's miss list (rows
// ascending, victim slots) is complete once the resolve kernel has published
// its copy_ready mark (== seq, after a fence; before the item's locations
// are written), and its staging entries once the mark carries no
// entries-pending bit, so the copy does not wait for the whole resolve
// grid.  CTA b owns items b, b + gridDim, ...: it takes, in order,
// every owned item whose mark is out as one batch (waiting, bounded, only
// when none is).  How its warps split the batch depends on c.steal:
//   - 0: the batch's rows form one flat list, four consecutive rows per warp
//     in turn (pinned regions past the GPU's translation reach, where a block
//     must keep to its own items' rows); an item joins a batch once its
//     staging entries are out too;
//   - 1: the warps claim each item's rows four at a time from the item's
//     claim cursor (zeroed by the resolve launch), the next claim in flight
//     while they copy, and a CTA whose own items are done then claims the
//     rows no CTA has claimed yet in the other items whose marks are out,
//     the next CTA's items first.  The copy blocks' speeds differ by SM and
//     the step waits for the last row.  An item is taken as soon as its
//     miss lists are out, its staging entries possibly still pending.
// A poll that runs out (after c.mark_polls polls; with 0 the marks are never
// read) falls back to waiting for the resolve grid.
constexpr int kBatchMax = 64;

template <int MAXI, bool kSmallRow, bool kSteal>
__global__ void __launch_bounds__(kCopyThreads)
    hostcopy_kernel(const __grid_constant__ CopyParams<MAXI> P) {
  __shared__ int s_n, s_next, s_wait;
  __shared__ int s_item[kBatchMax];
  __shared__ uint32_t s_pre[kBatchMax + 1];  // flat list: rows before each batch item
  const CopyCommon& c = P.c;
  const int tid = threadIdx.x, lane = tid & 31;
  // the gather may be launched now
  asm volatile("griddepcontrol.launch_dependents;");
  const uint32_t warp = (uint32_t)tid >> 5, nwarps = blockDim.x >> 5;
  const uint32_t want = c.seq & kSeqMask;
  bool waited = c.ready == nullptr, traced = false;
  if (waited) asm volatile("griddepcontrol.wait;" ::: "memory");
  // every unclaimed row of item j (cnt rows), kRowsPerWarp per claim: lane
  // 0's atomic, its result taken only after the current rows are copied.
  // The item's staging entries may still be pending when its rows are
  // claimed: before its first staging write the warp polls the mark (every
  // lane its own acquire, bounded) until the entries are out, or falls back
  // to waiting for the resolve grid.
  auto drain = [&](int j, uint32_t cnt) {
    const CopyItem& it = P.items[j];
    uint32_t* cur_p = c.cursor + it.pair;
    bool entries = waited;
    auto wait_entries = [&]() {
      for (uint32_t i = 0; !entries; ++i) {
        const uint32_t v = ld_acquire_u32(c.ready + it.pair);
        if (!(v & kMarkEntriesPending)) {
          entries = true;
        } else if (i >= c.mark_polls) {
          asm volatile("griddepcontrol.wait;" ::: "memory");
          waited = entries = true;
        } else {
          __nanosleep(256);
        }
      }
    };
    const uint32_t first = lane == 0 ? atomicAdd(cur_p, (uint32_t)kRowsPerWarp) : 0u;
    uint32_t cur = __shfl_sync(0xffffffffu, first, 0);
    while (cur < cnt) {
      const uint32_t pend = lane == 0 ? atomicAdd(cur_p, (uint32_t)kRowsPerWarp) : 0u;
      copy_rows<kSmallRow>(P, it, cur, min(cnt, cur + (uint32_t)kRowsPerWarp), lane,
                           wait_entries);
      cur = __shfl_sync(0xffffffffu, pend, 0);
    }
  };
  int next = blockIdx.x;
  bool had_rows = false;  // block-uniform: some owned item had misses
  for (;;) {
    if (tid == 0) {  // the next batch: owned items whose miss lists are out
      int n = 0, j = next, need_wait = 0;
      uint32_t acc = 0;
      while (j < c.n_items && n < kBatchMax) {
        const uint32_t* mark = c.ready + P.items[j].pair;
        const bool read = !waited && c.mark_polls != 0;
        // the claiming copy takes an item once its lists are out; the flat
        // list also needs its staging entries
        auto out = [&](uint32_t v) {
          return (v & kSeqMask) == want && (kSteal || !(v & kMarkEntriesPending));
        };
        uint32_t v = read ? ld_acquire_u32(mark) : 0u;
        bool ok = waited || (read && out(v));
        for (uint32_t i = 0; !ok && n == 0 && i < c.mark_polls; ++i) {
          __nanosleep(256);
          v = ld_acquire_u32(mark);
          ok = out(v);
        }
        if (!ok) {
          need_wait = n == 0;
          break;
        }
        s_item[n] = j;
        s_pre[n] = acc;
        // an item whose mark says "no misses" has written nothing to read
        acc += (v & kMarkNoMiss) ? 0u : c.miss_count[P.items[j].pair];
        ++n;
        j += gridDim.x;
      }
      s_pre[n] = acc;
      s_n = n;
      s_next = j;
      s_wait = need_wait;
    }
    __syncthreads();
    if (s_wait) {  // a mark never came: wait for the resolve grid, then go on
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
      __syncthreads();
      continue;
    }
    const int n = s_n, nxt = s_next;
    if (n == 0) break;
    if (!waited)  // each thread's own acquire of the batch's marks
      for (int b = 0; b < n; ++b) (void)ld_acquire_u32(c.ready + P.items[s_item[b]].pair);
    if (tid == 0 && !traced) {
      trace_mark(c.trace, kTraceCopy, false);  // copying starts
      traced = true;
    }
    had_rows = had_rows || s_pre[n] != 0;
    if constexpr (kSteal) {
      for (int b = 0; b < n; ++b) {
        const uint32_t cnt = s_pre[b + 1] - s_pre[b];
        if (cnt) drain(s_item[b], cnt);
      }
    } else {
      const int rb = c.row_bytes, cpr = rb >> 4;
      const uint32_t total = s_pre[n];
      for (uint32_t base = warp * kRowsPerWarp; base < total; base += nwarps * kRowsPerWarp) {
        const uint8_t* src[kRowsPerWarp];
        uint8_t* dst[kRowsPerWarp];
        // staging entries of the row (items whose host copy stages): the
        // entries e0 .. e1 of the item's miss_ent list, written at stg + e * rb
        uint8_t* stg[kRowsPerWarp];
        const int32_t* ents[kRowsPerWarp];
        int32_t e0[kRowsPerWarp], e1[kRowsPerWarp], itm[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          const uint32_t i = base + r;
          src[r] = nullptr;
          dst[r] = nullptr;
          stg[r] = nullptr;
          ents[r] = nullptr;
          e0[r] = e1[r] = 0;
          itm[r] = 0;
          if (i < total) {
            int lo = 0, hi = n - 1;  // last batch entry with s_pre <= i
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (s_pre[mid] <= i) lo = mid; else hi = mid - 1;
            }
            itm[r] = s_item[lo];
            const CopyItem& it = P.items[itm[r]];
            const uint32_t mi = i - s_pre[lo];
            const size_t off = (size_t)it.pair * c.Mcap + mi;
            const int32_t row = c.miss_rows[off];
            const int32_t slot = c.miss_slots[off];
            src[r] = it.host + (size_t)row * rb;
            dst[r] = c.hot + ((size_t)it.pair * c.B + slot) * rb;
            if (it.staging) {
              const int32_t* mo = c.miss_off + (size_t)it.pair * (c.Mcap + 1);
              stg[r] = it.staging;
              ents[r] = c.miss_ent + (size_t)it.pair * c.ent_cap;
              e0[r] = mo[mi];
              e1[r] = mo[mi + 1];
            }
          }
        }
        if (kSmallRow) {
          uint4 v[kRowsPerWarp][kChunksPerLane];
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int q = 0; q < kChunksPerLane; ++q) {
              const int ch = lane + 32 * q;
              if (src[r] && ch < cpr) v[r][q] = ld_sys(src[r] + ch * 16);
            }
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
#pragma unroll
            for (int q = 0; q < kChunksPerLane; ++q) {
              const int ch = lane + 32 * q;
              if (dst[r] && ch < cpr) *reinterpret_cast<uint4*>(dst[r] + ch * 16) = v[r][q];
            }
            // the same bytes to its staging entries, in the item's staging and
            // in that of the gather-only items sharing its locations
            const int ns = stg[r] ? P.items[itm[r]].nshare : 0;
            for (int k = e0[r]; k < e1[r]; ++k) {
              const size_t eo = (size_t)ents[r][k] * rb;
              for (int j = -1; j < ns; ++j) {
                uint8_t* to = (j < 0 ? stg[r] : P.items[itm[r]].share[j]) + eo;
#pragma unroll
                for (int q = 0; q < kChunksPerLane; ++q) {
                  const int ch = lane + 32 * q;
                  if (ch < cpr) *reinterpret_cast<uint4*>(to + ch * 16) = v[r][q];
                }
              }
            }
          }
        } else {
          for (int r = 0; r < kRowsPerWarp; ++r) {
            if (!src[r]) continue;
            const int ns = stg[r] ? P.items[itm[r]].nshare : 0;
            for (int ch = lane; ch < cpr; ch += 32) {
              const uint4 v = ld_sys(src[r] + ch * 16);
              *reinterpret_cast<uint4*>(dst[r] + ch * 16) = v;
              for (int k = e0[r]; k < e1[r]; ++k) {
                const size_t eo = (size_t)ents[r][k] * rb + ch * 16;
                *reinterpret_cast<uint4*>(stg[r] + eo) = v;
                for (int j = 0; j < ns; ++j)
                  *reinterpret_cast<uint4*>(P.items[itm[r]].share[j] + eo) = v;
              }
            }
          }
        }
      }
    }
    __syncthreads();  // the batch tables are rebuilt
    next = nxt;
  }
  // c.steal: the other items' unclaimed rows, the next CTA's items first: the
  // lanes test 32 items at a time with relaxed reads (a hint), then the warp
  // acquires each candidate's mark (every lane its own acquire) and drains it.
  // A block whose own items had no misses leaves at once instead: in a launch
  // with few or no misses (C8 has none) the gather wants its SM back, and the
  // scan would hold it about a microsecond longer for nothing.
  for (int base = 1; kSteal && (had_rows || (int)blockIdx.x >= c.n_items) && base < c.n_items;
       base += 32) {
    const int k = base + lane;
    int j = 0;
    bool cand = false;
    if (k < c.n_items) {
      j = (blockIdx.x + k) % c.n_items;
      const int pair = P.items[j].pair;
      const uint32_t v = waited ? want : ld_relaxed_u32(c.ready + pair);
      if ((v & kSeqMask) == want && !(v & kMarkNoMiss))
        cand = ld_relaxed_u32(c.cursor + pair) < ld_relaxed_u32(c.miss_count + pair);
    }
    for (uint32_t m = __ballot_sync(0xffffffffu, cand); m; m &= m - 1) {
      const int jj = __shfl_sync(0xffffffffu, j, __ffs(m) - 1);
      const int pair = P.items[jj].pair;
      if (!waited) (void)ld_acquire_u32(c.ready + pair);
      drain(jj, c.miss_count[pair]);
    }
  }
  // this grid completes only after the resolve grid (the gather and the
  // fresh-row copy rely on that): its last block waits for it.  The others
  // leave once no row is left to copy; each holds a whole SM's registers
  // (512 threads x 128), which the gather can use as soon as it is gone.
  if (!waited && blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  if (tid == 0) trace_mark(c.trace, kTraceCopy, true);
}

template <int MAXI>
cudaError_t launch_t(const CopyCommon& c, const CopyItem* items, int n, int ctas, int threads,
                     bool pdl, size_t hold_smem, cudaStream_t stream) {
  CopyParams<MAXI> P;
  P.c = c;
  P.c.n_items = n;
  for (int i = 0; i < n; ++i) P.items[i] = items[i];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = hold_smem;  // unused by the kernel: keeps other CTAs off its SM
  cfg.stream = stream;
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const bool small = (c.row_bytes >> 4) <= 32 * kChunksPerLane;
  if (c.steal)
    return small ? cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, true, true>, P)
                 : cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, false, true>, P);
  return small ? cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, true, false>, P)
               : cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, false, false>, P);
}

// ---------------------------------------------------------------- page moves

struct PageMoveParams {
  int32_t n;
  int32_t page_bytes;
  PageMove m[kPageMovesMax];
};
static_assert(sizeof(PageMoveParams) <= 32764, "page list too large");

// Grid-stride over the 16-byte chunks of every listed page; each thread
// keeps four chunks in flight so the link sees enough outstanding requests
// (one side of every move is mapped host memory).
__global__ void __launch_bounds__(kPageMoveThreads)
    page_move_kernel(const __grid_constant__ PageMoveParams P) {
  const uint32_t cpp = (uint32_t)P.page_bytes >> 4;  // chunks per page
  const uint32_t total = (uint32_t)P.n * cpp;
  const uint32_t stride = gridDim.x * blockDim.x;
  constexpr int kIn = 4;
  for (uint32_t base = blockIdx.x * blockDim.x + threadIdx.x; base < total;
       base += stride * kIn) {
    uint4 v[kIn];
#pragma unroll
    for (int u = 0; u < kIn; ++u) {
      const uint32_t ch = base + u * stride;
      if (ch < total) {
        const uint32_t pg = ch / cpp, c = ch - pg * cpp;
        v[u] = __ldcs(reinterpret_cast<const uint4*>(P.m[pg].src) + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kIn; ++u) {
      const uint32_t ch = base + u * stride;
      if (ch < total) {
        const uint32_t pg = ch / cpp, c = ch - pg * cpp;
        __stcs(reinterpret_cast<uint4*>(P.m[pg].dst) + c, v[u]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_page_moves(const PageMove* moves, int n, int page_bytes, int ctas,
                              cudaStream_t stream) {
  for (int b = 0; b < n; b += kPageMovesMax) {
    PageMoveParams P;
    P.n = std::min(kPageMovesMax, n - b);
    P.page_bytes = page_bytes;
    for (int i = 0; i < P.n; ++i) P.m[i] = moves[b + i];
    const int64_t chunks = (int64_t)P.n * (page_bytes >> 4);
    const int64_t need = (chunks + kPageMoveThreads - 1) / kPageMoveThreads;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ctas, need));
    page_move_kernel<<<grid, kPageMoveThreads, 0, stream>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t hostcopy_set_carveout(size_t hold_smem) {
  for (const void* k : {(const void*)hostcopy_kernel<kCopyItemsMax, true, false>,
                        (const void*)hostcopy_kernel<kCopyItemsMax, false, false>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, true, false>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, false, false>,
                        (const void*)hostcopy_kernel<kCopyItemsMax, true, true>,
                        (const void*)hostcopy_kernel<kCopyItemsMax, false, true>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, true, true>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, false, true>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hold_smem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_hostcopy(const CopyCommon& c, const CopyItem* items, int n_items,
                            int ctas, int threads, bool pdl, size_t hold_smem,
                            cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (n_items > kCopyItemsMax || n_items > kCopyThreads) return cudaErrorInvalidValue;
  if (threads < 32 || threads > kCopyThreads || threads % 32) return cudaErrorInvalidValue;
  // the whole table travels with every launch: a small one for small steps
  if (n_items <= kCopyItemsSmall)
    return launch_t<kCopyItemsSmall>(c, items, n_items, ctas, threads, pdl, hold_smem, stream);
  return launch_t<kCopyItemsMax>(c, items, n_items, ctas, threads, pdl, hold_smem, stream);
}

}  // namespace dhs
