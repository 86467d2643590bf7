// Host-copy kernel: step 3 of resolution ("a copy from pinned host memory
// into the hot cache"; "Adaptive DHiSparse", How it works / Resolution).
//
// Reads the missing rows straight out of mapped pinned host memory over
// NVLink-C2C into their victim hot-cache slots.  The pages note that the
// copy kernel scales from 4 to 32 thread blocks with batch size; on GB300
// fewer than about 16 blocks leave the host link idle, so the grid is at
// least the upper end, 32 blocks, whatever the batch.  The pool grows it
// further when the items' pinned regions are large (each block's share
// kept within about 1 GiB, so that the translations of its rows stay cached
// near its SM).  Past 16 GiB of pinned rows it launches the copy after the
// resolve grid, so that block b lands on the same SM every step, unless every
// copy block finds an SM that the resolve grid leaves free.  Each warp keeps up
// to four 1152-byte rows in flight (12 x 16-byte loads per lane) so the link
// sees enough outstanding requests to cover its latency.
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

// Copy the miss rows of the launch's items.  CTA b owns items b, b + gridDim,
// ...  An item's miss list (rows ascending, victim slots, staging entries)
// is complete once the resolve kernel has published its copy_ready mark
// (== seq, after a fence; before the item's locations are written), so the
// CTA does not wait for the whole resolve grid: it
// takes, in order, every owned item whose mark is out as one batch (waiting,
// bounded, only when none is), and its warps copy the batch's rows as one
// flat list, four rows per warp in flight.  A poll that runs out (after
// c.mark_polls polls; with 0 the marks are never read) falls back to waiting
// for the resolve grid.
constexpr int kBatchMax = 64;

template <int MAXI, bool kSmallRow>
__global__ void __launch_bounds__(kCopyThreads)
    hostcopy_kernel(const __grid_constant__ CopyParams<MAXI> P) {
  __shared__ int s_n, s_next, s_wait;
  __shared__ int s_item[kBatchMax];
  __shared__ uint32_t s_pre[kBatchMax + 1];
  const CopyCommon& c = P.c;
  const int tid = threadIdx.x, lane = tid & 31;
  // the gather may be launched now
  asm volatile("griddepcontrol.launch_dependents;");
  const int rb = c.row_bytes;
  const int cpr = rb >> 4;
  const uint32_t warp = (uint32_t)tid >> 5, nwarps = blockDim.x >> 5;
  const uint32_t want = c.seq & kSeqMask;
  bool waited = c.ready == nullptr, traced = false;
  if (waited) asm volatile("griddepcontrol.wait;" ::: "memory");
  int next = blockIdx.x;
  for (;;) {
    if (tid == 0) {  // the next batch: owned items whose miss lists are out
      int n = 0, j = next, need_wait = 0;
      uint32_t acc = 0;
      while (j < c.n_items && n < kBatchMax) {
        const uint32_t* mark = c.ready + P.items[j].pair;
        const bool read = !waited && c.mark_polls != 0;
        uint32_t v = read ? ld_acquire_u32(mark) : 0u;
        bool ok = waited || (read && (v & kSeqMask) == want);
        for (uint32_t i = 0; !ok && n == 0 && i < c.mark_polls; ++i) {
          __nanosleep(256);
          v = ld_acquire_u32(mark);
          ok = (v & kSeqMask) == want;
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
    __syncthreads();  // the batch tables are rebuilt
    next = nxt;
  }
  // this grid completes only after the resolve grid (the gather and the
  // fresh-row copy rely on that): its last block waits for it.  The others
  // leave once their items are copied; each holds a whole SM's registers
  // (512 threads x 128), which the gather can use as soon as it is gone.
  if (!waited && blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  __syncthreads();
  if (tid == 0) trace_mark(c.trace, kTraceCopy, true);
}

template <int MAXI>
cudaError_t launch_t(const CopyCommon& c, const CopyItem* items, int n, int ctas,
                     bool pdl, cudaStream_t stream) {
  CopyParams<MAXI> P;
  P.c = c;
  P.c.n_items = n;
  for (int i = 0; i < n; ++i) P.items[i] = items[i];
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kCopyThreads);
  cfg.stream = stream;
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if ((c.row_bytes >> 4) <= 32 * kChunksPerLane)
    return cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, true>, P);
  return cudaLaunchKernelEx(&cfg, hostcopy_kernel<MAXI, false>, P);
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

cudaError_t hostcopy_set_carveout() {
  for (const void* k : {(const void*)hostcopy_kernel<kCopyItemsMax, true>,
                        (const void*)hostcopy_kernel<kCopyItemsMax, false>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, true>,
                        (const void*)hostcopy_kernel<kCopyItemsSmall, false>}) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_hostcopy(const CopyCommon& c, const CopyItem* items, int n_items,
                            int ctas, bool pdl, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (n_items > kCopyItemsMax || n_items > kCopyThreads) return cudaErrorInvalidValue;
  // the whole table travels with every launch: a small one for small steps
  if (n_items <= kCopyItemsSmall)
    return launch_t<kCopyItemsSmall>(c, items, n_items, ctas, pdl, stream);
  return launch_t<kCopyItemsMax>(c, items, n_items, ctas, pdl, stream);
}

}  // namespace dhs
