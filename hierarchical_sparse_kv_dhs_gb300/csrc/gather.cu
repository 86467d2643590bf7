// Gather kernels: staging[item][q][i] = the KV row at loc[item][q][i].
//
// "Adaptive DHiSparse", How it works: selected rows are consumed by sparse
// attention from verification staging; Reuse layers gather an inherited
// location vector.  This is the byte-dominant step of the decode path
// (1152 bytes read + 1152 written per entry against 4 bytes of location), a
// pure HBM copy, so it is built for memory-level parallelism, not arithmetic.
// One CTA per tile of entries of one item; two implementations:
//   * TMA (default): 16 entries per CTA, split between two warps of 8; lane
//     e of a warp moves its entry with one bulk copy (cp.async.bulk) global
//     -> shared, completion counted on the warp's own mbarrier, then one bulk
//     copy shared -> staging.  No row byte passes through registers; eleven
//     18 KB tiles stay in flight per SM.
//   * vector: 256 threads per tile of 32 entries, 9 x 16-byte loads in flight
//     per thread, consecutive threads on consecutive 16-byte chunks
//     (full-line coalesced).
//
// Early phase (fused resolve + gather).  A row that resolves in step 1 of
// "Resolution" -- the tail (row >= L - T) or a ready optional page -- has a
// location that is a pure function of the row, L, T and the page map, none of
// which the resolve kernel of the same step changes.  The fused launch
// (programmatic dependent launch) therefore copies those rows while the
// resolve kernel still runs, and only tiles with rows that need the hot cache
// wait for the item's locations (or the resolve / host-copy grids).  Step-1
// rows never wait for the item's outcome: a failed resolution still gives
// them their locations (it changes no state they depend on), and every other
// entry of a failed item has none, so its rows become zeros.
#include <algorithm>

#include "dhs_internal.h"

namespace dhs {
namespace {

template <int MAXI>
struct GatherParams {
  GatherCommon c;
  GatherItem items[MAXI];
};
// kernel parameter space holds at most 32764 bytes
static_assert(sizeof(GatherParams<kGatherItemsLarge>) <= 32764, "gather item table too large");

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait (whole warp) until the resolve kernel has published the
// item's locations; false if they did not come out within c.mark_polls polls
// -- the caller then waits for the resolve / host-copy grids instead, so
// giving up costs time, never correctness.  Every lane takes its own acquire.
__device__ __forceinline__ bool wait_loc_ready(const GatherCommon& c, const GatherItem& it) {
  const uint32_t want = it.seq & kSeqMask;
  for (uint32_t i = 0; i < c.mark_polls; ++i) {
    const bool r = ld_acquire(&c.loc_ready[it.pair]) == want;
    if (__all_sync(0xFFFFFFFFu, r)) return true;
    __nanosleep(200);
  }
  return false;
}

// True if `loc` names a hot slot that this step's host copy fills.
__device__ __forceinline__ bool fresh_loc(const GatherCommon& c, uint32_t loc) {
  if ((loc >> 30) != kTierHot || loc == kNoLoc || loc == kEndLoc) return false;
  const uint32_t idx = loc & 0x3FFFFFFFu;
  if (idx >= c.hot_rows) return false;  // invalid: the copy reports it
  const uint32_t pair = idx / (uint32_t)c.B, slot = idx - pair * (uint32_t)c.B;
  return (ld_relaxed(&c.fill[(size_t)pair * c.fill_words + (slot >> 5)]) >> (slot & 31)) & 1u;
}

template <int MAXI>
__device__ __forceinline__ int find_item(const GatherParams<MAXI>& P, int tile) {
  if (P.c.item_tiles > 0) return tile / P.c.item_tiles;  // equal items: no search
  int lo = 0, hi = P.c.n_items - 1;  // last item whose first tile <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.items[mid].tile0 <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Decode one location to a source row pointer (nullptr: write zeros).
__device__ __forceinline__ const uint8_t* row_ptr(const GatherCommon& c, uint32_t loc) {
  if (loc == kNoLoc) return nullptr;
  const uint32_t tier = loc >> 30, idx = loc & 0x3FFFFFFFu;
  const uint8_t* base = nullptr;
  uint32_t lim = 0;
  if (tier == kTierTail) { base = c.tail; lim = c.tail_rows; }
  else if (tier == kTierOpt) { base = c.opt; lim = c.opt_rows; }
  else if (tier == kTierHot) { base = c.hot; lim = c.hot_rows; }
  if (!base || idx >= lim) {
    atomicOr(c.status, kStatusEloc);
    return nullptr;
  }
  return base + (size_t)idx * c.row_bytes;
}

// Step-1 row address of `row` of an item, or nullptr if the row needs the
// hot cache or is out of range (which the resolve kernel reports).  A row
// appended by this launch is in the tail once the resolve kernel has written
// it there; until then the same bytes are in the append's source rows.
__device__ __forceinline__ const uint8_t* step1_ptr(const GatherCommon& c,
                                                    const GatherItem& it, int32_t row) {
  if (row < 0) return nullptr;
  if ((int64_t)row >= it.L0) {
    if (!it.app || (int64_t)row >= it.L) return nullptr;
    return it.app + (size_t)((int64_t)row - it.L0) * c.row_bytes;
  }
  const int64_t T = c.T;
  if ((int64_t)row >= it.L - T)
    return c.tail + ((size_t)it.pair * T + (size_t)((int64_t)row % T)) * c.row_bytes;
  const int ps = c.page_shift;
  const int64_t page = (int64_t)row >> ps;
  if (((page + 1) << ps) > it.N) return nullptr;
  const int32_t slot = c.map[(size_t)it.pair * c.Pmax + page];
  if (slot < 0) return nullptr;
  const int64_t idx = ((int64_t)slot << ps) + (row & (((int64_t)1 << ps) - 1));
  return c.opt + (size_t)idx * c.row_bytes;
}

// End of a gather CTA.  The gather grid must not complete before the resolve
// / host-copy grids it overlaps (stream order for whatever follows), so its
// last block waits for them; every other CTA leaves as soon as its rows are
// written.
// DHS_OPT_TRACE marks of the gather: one CTA in 64, and the last.  C64's
// 262,144 CTAs all marking two shared words slowed the traced steps' host
// copy by a fifth; the sampled first start and last end are within a CTA's
// lifetime of the true ones.
__device__ __forceinline__ bool trace_sampled() {
  return (blockIdx.x & 63u) == 0 || blockIdx.x == gridDim.x - 1;
}

__device__ __forceinline__ void end_grid(const GatherCommon& c) {
  if (blockIdx.x == gridDim.x - 1) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (c.trace) __syncthreads();  // the CTA's end is its last warp's end
  if (threadIdx.x == 0 && trace_sampled()) trace_mark(c.trace, kTraceGather, true);
}

// ---------------------------------------------------------------- vector variant

// Copy the entries of the tile whose s_phase equals `phase`.
template <int CPR>
__device__ __forceinline__ void copy_tile(const GatherCommon& c, uint8_t* dst,
                                          const uint8_t* const* s_src,
                                          const uint8_t* s_phase, int ne, int phase) {
  const int tid = threadIdx.x;
  if constexpr (CPR != 0) {
    constexpr int U = (kGatherTileRows * CPR + kGatherThreads - 1) / kGatherThreads;
    const int total = ne * CPR;
    uint4 v[U];
    uint32_t take = 0;  // bit u: chunk u belongs to this phase
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = tid + u * kGatherThreads;
      if (ch < total) {
        const int e = ch / CPR, p = ch - e * CPR;
        if (s_phase[e] == phase) {
          const uint8_t* s = s_src[e];
          v[u] = s ? ld_stream(s + p * 16) : make_uint4(0u, 0u, 0u, 0u);
          take |= 1u << u;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if ((take >> u) & 1u)
        *reinterpret_cast<uint4*>(dst + (size_t)(tid + u * kGatherThreads) * 16) = v[u];
    }
  } else {
    const int cpr = c.row_bytes >> 4;
    const int total = ne * cpr;
    for (int ch = tid; ch < total; ch += kGatherThreads) {
      const int e = ch / cpr, p = ch - e * cpr;
      if (s_phase[e] != phase) continue;
      const uint8_t* s = s_src[e];
      const uint4 v = s ? ld_stream(s + p * 16) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dst + (size_t)ch * 16) = v;
    }
  }
}

// CPR = 16-byte chunks per row (0: runtime value).
template <int MAXI, int CPR>
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const __grid_constant__ GatherParams<MAXI> P) {
  __shared__ const uint8_t* s_src[kGatherTileRows];
  __shared__ uint8_t s_phase[kGatherTileRows];
  const GatherCommon& c = P.c;
  const int tile = blockIdx.x;
  const GatherItem& it = P.items[find_item(P, tile)];
  const int e0 = (tile - it.tile0) * kGatherTileRows;
  const int ne = min(kGatherTileRows, it.n - e0);
  const int tid = threadIdx.x;
  uint8_t* dst = it.staging + (size_t)e0 * c.row_bytes;
  const bool early = c.early && it.sel != nullptr;
  asm volatile("griddepcontrol.launch_dependents;");
  if (tid == 0 && trace_sampled()) trace_mark(c.trace, kTraceGather, false);

  // phase 0: rows resolved in step 1 (fused launch only)
  int deferred = 0;
  if (tid < ne) {
    const uint8_t* p = early ? step1_ptr(c, it, it.sel[e0 + tid]) : nullptr;
    s_src[tid] = p;
    s_phase[tid] = p ? 0 : 1;
    deferred = p == nullptr;
  }
  const int any_deferred = __syncthreads_or(deferred);
  if (early) copy_tile<CPR>(c, dst, s_src, s_phase, ne, 0);
  if (any_deferred) {
    // rows that needed the hot cache (or no early phase): wait for the
    // resolve / host-copy grids (a no-op without programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid < ne && s_phase[tid] == 1) {
      const uint32_t l = it.loc[e0 + tid];
      if (l == kEndLoc) s_phase[tid] = 2;  // past a union list: nothing to write
      else s_src[tid] = row_ptr(c, l);
    }
    __syncthreads();
    copy_tile<CPR>(c, dst, s_src, s_phase, ne, 1);
  }
  end_grid(c);
}

// ---------------------------------------------------------------- TMA variant

constexpr int kTmaThreads = 32 * kTmaWarps;
constexpr uint32_t kWaitPolls = 1u << 26;  // bounded mbarrier wait

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}"
      ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Wait for the mbarrier phase with the given parity; false if it never came.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

// The same load, its row marked first to leave L2: a row that nothing else
// in the launch reads then gives way before the staging rows just written.
__device__ __forceinline__ void bulk_load_once(void* smem_dst, const void* gsrc,
                                               uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], pol;\n\t}"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
               ::"l"(gdst), "r"(smem_u32(smem_src)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int MAXI>
__global__ void __launch_bounds__(kTmaThreads)
    gather_tma_kernel(const __grid_constant__ GatherParams<MAXI> P) {
  extern __shared__ __align__(128) uint8_t s_rows[];  // [kTmaTileRows][row_bytes]
  __shared__ __align__(8) uint64_t s_bars[kTmaWarps];
  const GatherCommon& c = P.c;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rb = (uint32_t)c.row_bytes;
  uint64_t& s_bar = s_bars[warp];
  // lanes past the warp's rows hold none (their entries never exist)
  uint8_t* my_row = s_rows + (size_t)(warp * kTmaWarpRows + min(lane, kTmaWarpRows - 1)) * rb;
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0 && trace_sampled()) trace_mark(c.trace, kTraceGather, false);
  if (lane == 0) mbar_init(&s_bar, 1);
  __syncwarp();
  uint32_t parity = 0;
  bool stored = false, ok = true, waited = false;
  uint8_t* dst = nullptr;

  // Move entry `lane` (src: row address, nullptr = zeros) to `dst` when
  // `mine`; false if the bounded wait gave up.
  auto move = [&](bool mine, const uint8_t* src) -> bool {
    const bool load = mine && src != nullptr;
    const unsigned lmask = __ballot_sync(0xFFFFFFFFu, load);
    if (mine && !load) {  // zeros: plain stores, then hand over to the async proxy
      for (uint32_t o = 0; o < rb; o += 16)
        *reinterpret_cast<uint4*>(my_row + o) = make_uint4(0u, 0u, 0u, 0u);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (lmask) {
      if (lane == 0) mbar_arrive_expect(&s_bar, (uint32_t)__popc(lmask) * rb);
      __syncwarp();
      if (load) {
        if (c.read_once) bulk_load_once(my_row, src, rb, &s_bar);
        else bulk_load(my_row, src, rb, &s_bar);
      }
      // one answer for the whole warp, so every later warp collective is
      // reached by all lanes
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&s_bar, parity))) {
        if (lane == 0) atomicOr(c.status, kStatusEtimeout);
        return false;
      }
      parity ^= 1u;
    }
    __syncwarp();
    if (mine) {
      bulk_store(dst, my_row, rb);
      stored = true;
    }
    return true;
  };

  // c.tpc consecutive tiles per CTA (one by default)
  for (int t = 0; t < c.tpc && ok; ++t) {
    const int tile = blockIdx.x * c.tpc + t;
    if (tile >= c.n_tiles) break;
    // the previous tile's stores must have read its rows out of shared memory
    if (stored) {
      asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      stored = false;
    }
    const GatherItem& it = P.items[find_item(P, tile)];
    // this warp's entries of the tile (none past the end of the item)
    const int e0 = (tile - it.tile0) * kTmaTileRows + warp * kTmaWarpRows;
    const int ne = min(kTmaWarpRows, it.n - e0);
    if (ne <= 0) continue;
    dst = it.staging + ((size_t)e0 + lane) * rb;
    const bool early = c.early && it.sel != nullptr;

    const uint8_t* src = nullptr;
    if (early && lane < ne) src = step1_ptr(c, it, it.sel[e0 + lane]);
    bool deferred = lane < ne && src == nullptr;
    if (early) ok = move(src != nullptr, src);  // rows resolved in step 1
    const bool lr = c.early && (it.flags & kGiLocReady) && !waited;
    if (ok && __any_sync(0xFFFFFFFFu, deferred) && lr && wait_loc_ready(c, it)) {
      // the item's locations are out: every row but the fresh ones (hot slots
      // the host copy is still filling) can move now
      const uint32_t l = deferred ? ld_relaxed(&it.loc[e0 + lane]) : kEndLoc;
      const bool fresh = deferred && fresh_loc(c, l);
      const bool now = deferred && l != kEndLoc && !fresh;
      ok = move(now, now ? row_ptr(c, l) : nullptr);
      // the host copy writes a staged item's fresh rows into staging itself
      bool later = fresh && !(it.flags & kGiStaged);
      if (c.later) {  // hand the fresh rows to the list copied after the copy grid
        const unsigned fm = __ballot_sync(0xFFFFFFFFu, later);
        uint32_t base = 0;
        if (lane == 0 && fm) base = atomicAdd(&c.later_count[c.gen & 1u], (uint32_t)__popc(fm));
        base = __shfl_sync(0xFFFFFFFFu, base, 0);
        const uint32_t cnt = (uint32_t)__popc(fm);
        const bool fits = (uint64_t)base + cnt <= c.later_cap;
        const uint32_t slot = base + (uint32_t)__popc(fm & ((1u << lane) - 1u));
        if (later && fits) {
          c.later[slot].dst = dst;
          c.later[slot].loc = l;
          later = false;
        } else if (later && slot < c.later_cap) {
          c.later[slot].dst = nullptr;  // the list is full: the tile copies it
        }
      }
      deferred = later;
    }
    if (ok && __any_sync(0xFFFFFFFFu, deferred)) {
      // rows that needed the hot cache (or no early phase): wait for the
      // resolve / host-copy grids (a no-op without programmatic dependent launch)
      if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
      const uint32_t l = deferred ? it.loc[e0 + lane] : kEndLoc;
      const bool live = l != kEndLoc;  // past a union list: nothing to write
      ok = move(live, live ? row_ptr(c, l) : nullptr);
    }
  }
  // shared memory must outlive the stores' reads
  if (stored) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  end_grid(c);
}

// ---------------------------------------------------------------- fresh rows

// Copy the fresh-row list of this generation (hot slot -> staging) once the
// gather grid -- whose last block waits for the host-copy grid -- is done.
// Each warp keeps four rows in flight, as the host copy does.
__global__ void __launch_bounds__(kLaterThreads) gather_later_kernel(const GatherCommon c) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) trace_mark(c.trace, kTraceLater, false);  // copying starts
  const uint32_t total = min(c.later_count[c.gen & 1u], c.later_cap);
  const int lane = threadIdx.x & 31;
  const int cpr = c.row_bytes >> 4;
  const uint32_t gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * blockDim.x) >> 5;
  constexpr int kRows = 4;
  for (uint32_t base = gwarp * kRows; base < total; base += nwarps * kRows) {
    for (int r = 0; r < kRows; ++r) {
      const uint32_t i = base + r;
      if (i >= total) break;
      uint8_t* dst = c.later[i].dst;
      if (!dst) continue;
      const uint8_t* src = row_ptr(c, c.later[i].loc);
      for (int ch = lane; ch < cpr; ch += 32) {
        const uint4 v = src ? *reinterpret_cast<const uint4*>(src + ch * 16)
                            : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(dst + ch * 16) = v;
      }
    }
  }
  if (threadIdx.x == 0) trace_mark(c.trace, kTraceLater, true);
}

template <int MAXI>
cudaError_t launch_t(const GatherCommon& c, const GatherItem* items, int n, bool pdl,
                     int impl, cudaStream_t stream) {
  GatherParams<MAXI> P;
  P.c = c;
  P.c.n_items = n;
  for (int i = 0; i < n; ++i) P.items[i] = items[i];
  if (c.n_tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)c.n_tiles);
  cfg.stream = stream;
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  if (impl == kGatherTma) {
    cfg.gridDim = dim3((unsigned)((c.n_tiles + c.tpc - 1) / c.tpc));
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = (size_t)kTmaTileRows * c.row_bytes;
    return cudaLaunchKernelEx(&cfg, gather_tma_kernel<MAXI>, P);
  }
  cfg.blockDim = dim3(kGatherThreads);
  if (c.row_bytes == 1152) return cudaLaunchKernelEx(&cfg, gather_kernel<MAXI, 72>, P);
  return cudaLaunchKernelEx(&cfg, gather_kernel<MAXI, 0>, P);
}

}  // namespace

cudaError_t launch_gather_later(const GatherCommon& c, int ctas, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kLaterThreads);
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_later_kernel, c);
}

cudaError_t gather_set_carveout() {
  const void* ks[] = {(const void*)gather_kernel<kGatherItemsSmall, 72>,
                      (const void*)gather_kernel<kGatherItemsSmall, 0>,
                      (const void*)gather_kernel<kGatherItemsLarge, 72>,
                      (const void*)gather_kernel<kGatherItemsLarge, 0>,
                      (const void*)gather_tma_kernel<kGatherItemsSmall>,
                      (const void*)gather_tma_kernel<kGatherItemsLarge>};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t gather_set_smem_limit(int row_bytes, int optin, bool* tma_ok) {
  const int bytes = kTmaTileRows * row_bytes;
  *tma_ok = bytes + 1024 <= optin;  // 1 KB for the kernel's static shared memory
  if (!*tma_ok || bytes <= 48 * 1024) return cudaSuccess;
  for (const void* f : {(const void*)gather_tma_kernel<kGatherItemsSmall>,
                        (const void*)gather_tma_kernel<kGatherItemsLarge>}) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_gather(const GatherCommon& c, const GatherItem* items, int n_items,
                          bool pdl, int impl, cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (n_items <= kGatherItemsSmall)
    return launch_t<kGatherItemsSmall>(c, items, n_items, pdl, impl, stream);
  if (n_items <= kGatherItemsLarge)
    return launch_t<kGatherItemsLarge>(c, items, n_items, pdl, impl, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dhs
