// Gather kernel: staging[item][q][i] = the KV row at loc[item][q][i].
//
// "Adaptive DHiSparse", How it works: selected rows are consumed by sparse
// attention from verification staging; Reuse layers gather an inherited
// location vector.  This is the byte-dominant step of the decode path (2 x
// 1152 bytes per entry against 4 bytes of location), a pure HBM copy, so it
// is built for coalescing, not arithmetic:
//   * one CTA per tile of 32 entries of one item; the 32 row addresses are
//     resolved once into shared memory (tier -> arena, bounds-checked);
//   * the tile is 32 x 72 chunks of 16 bytes = 2304 chunks = 9 per thread;
//     consecutive threads read consecutive 16-byte chunks of a row (each
//     1152-byte row is nine whole 128-byte lines) and write consecutive
//     chunks of the contiguous staging tile, so every load and store is a
//     full-line coalesced access;
//   * all nine loads are issued before the first store (36 KB in flight per
//     CTA) to cover HBM latency; loads use the non-coherent no-allocate path.
//
// Early phase (fused resolve + gather only).  Where a row resolves in step 1
// of "Resolution" -- the tail (row >= L - T) or a ready optional page -- its
// location is a pure function of the row, L, T and the page map, none of
// which the resolve kernel of the same step changes.  The fused launch
// therefore copies those rows at once, while the resolve and host-copy
// kernels still run (programmatic dependent launch), and waits for them
// (griddepcontrol.wait) only before rows that need the hot cache.  After the
// wait a tile re-checks its item's resolve status: a failed item (row out of
// range, budget overflow) gets zeros everywhere, exactly as without the
// early phase.
#include "dhs_internal.h"

namespace dhs {
namespace {

template <int MAXI>
struct GatherParams {
  GatherCommon c;
  GatherItem items[MAXI];
};

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int MAXI>
__device__ __forceinline__ int find_item(const GatherParams<MAXI>& P, int tile) {
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
// hot cache (or is out of range, which the resolve kernel reports).
__device__ __forceinline__ const uint8_t* step1_ptr(const GatherCommon& c,
                                                    const GatherItem& it, int32_t row) {
  if (row < 0 || (int64_t)row >= it.L0) return nullptr;  // incl. rows appended now
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

// After the whole grid has written its rows: the last CTA to finish (an
// atomic ticket, no waiting on other CTAs) waits for the resolve / host-copy
// grids -- so the gather grid never completes before them -- zeroes the
// staging of every early item whose resolution failed (its step-1 rows may
// already have been copied), and resets the ticket for the next launch.
template <int MAXI>
__device__ void finish_grid(const GatherParams<MAXI>& P) {
  const GatherCommon& c = P.c;
  __shared__ int s_last;
  __threadfence();  // this CTA's staging writes are visible before its ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    s_last = atomicAdd(c.done, 1u) == gridDim.x - 1;
    trace_mark(c.trace, kTraceGather, true);
  }
  __syncthreads();
  if (!s_last) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __threadfence();
  if (c.early) {
    for (int i = 0; i < c.n_items; ++i) {
      const GatherItem& it = P.items[i];
      if (!it.sel || c.pair_status[it.pair] == 0) continue;
      uint4* d = reinterpret_cast<uint4*>(it.staging);
      const size_t chunks = (size_t)it.n * (c.row_bytes >> 4);
      for (size_t j = threadIdx.x; j < chunks; j += blockDim.x) d[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (threadIdx.x == 0) {
    *c.done = 0u;
    trace_mark(c.trace, kTraceGather, true);
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
  if (tid == 0) trace_mark(c.trace, kTraceGather, false);
  uint8_t* dst = it.staging + (size_t)e0 * c.row_bytes;
  const bool early = c.early && it.sel != nullptr;

  // phase 0: rows resolved in step 1 (fused launch only)
  int deferred = 0;
  if (tid < ne) {
    const uint8_t* p = early ? step1_ptr(c, it, it.sel[e0 + tid]) : nullptr;
    s_src[tid] = p;
    s_phase[tid] = p ? 0 : 1;
    deferred = p == nullptr;
  }
  const int any_deferred = __syncthreads_or(deferred);
#pragma unroll 1
  for (int ph = early ? 0 : 1; ph < 2; ++ph) {
    if (ph == 1) {
      if (!any_deferred) break;
      // rows that needed the hot cache: wait for the resolve / host-copy grids
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (tid < ne && s_phase[tid] == 1) s_src[tid] = row_ptr(c, it.loc[e0 + tid]);
      __syncthreads();
    }
    copy_tile<CPR>(c, dst, s_src, s_phase, ne, ph);
  }
  finish_grid(P);
}

// ---------------------------------------------------------------- TMA variant
// One warp per 32-entry tile: lane e moves entry e with one bulk copy
// (cp.async.bulk) global -> shared, completion counted on an mbarrier, then
// one bulk copy shared -> staging.  No row bytes pass through registers, so
// 6 tiles (36 KB each) stay in flight per SM with 32 threads apiece.
constexpr int kTmaThreads = 32;
constexpr int kTmaMaxLocal = 256;  // tiles per warp (deferred-lane masks in shared memory)

__host__ __device__ inline size_t tma_smem_bytes(int row_bytes) {
  return 2 * (size_t)kGatherTileRows * row_bytes + kTmaMaxLocal * sizeof(uint32_t);
}
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

__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Persistent, double-buffered, software-pipelined.  The launch's entries
// (all items back to back) are split evenly over the warps; warp b moves its
// range in chunks of 32 rows (lane l: entry chunk_start + l, each lane finds
// its own item, so a chunk may straddle items).  Four chunks are in the pipe:
// the bulk copies of chunk i land in one buffer while chunk i+1's bulk loads
// fill the other, chunk i+2's row addresses are computed (for step-1 rows:
// one page-map read) and chunk i+3's selection / location entries are loaded,
// so address latency overlaps data movement.  With the early phase on, pass 0
// moves the step-1 rows and records, per chunk, the lanes still waiting for
// the hot cache; after one griddepcontrol.wait, pass 1 moves only those.
struct TmaSlot {
  const uint8_t* src;  // row to load (nullptr: zeros)
  uint8_t* dst;        // staging row
  bool mine;           // this lane moves a row in this chunk
  unsigned lmask;      // lanes with a bulk load in flight
};

template <int MAXI>
__device__ __forceinline__ int find_item_entry(const GatherParams<MAXI>& P, int g) {
  int lo = 0, hi = P.c.n_items - 1;  // last item whose first entry <= g
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.items[mid].ent0 <= g) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int MAXI>
__global__ void __launch_bounds__(kTmaThreads)
    gather_tma_kernel(const __grid_constant__ GatherParams<MAXI> P) {
  extern __shared__ __align__(128) uint8_t s_dyn[];  // [2][32][rb], then chunk masks
  __shared__ __align__(8) uint64_t s_bar[2];
  const GatherCommon& c = P.c;
  const int lane = threadIdx.x;
  const uint32_t rb = (uint32_t)c.row_bytes;
  const size_t buf_bytes = (size_t)kGatherTileRows * rb;
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_dyn + 2 * buf_bytes);
  if (lane == 0) {
    trace_mark(c.trace, kTraceGather, false);
    if (c.trace) {  // mean warp start, relative to the resolve kernel's start
      const unsigned long long t0 = *(volatile unsigned long long*)&c.trace[0];
      atomicAdd(&c.trace[6], trace_now() - t0);
      atomicAdd(&c.trace[7], 1ull);
    }
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
  }
  __syncwarp();
  // this warp's entries [lo, hi)
  const int64_t E = c.n_entries, G = gridDim.x;
  const int lo = (int)(E * blockIdx.x / G), hi = (int)(E * (blockIdx.x + 1) / G);
  const int n_local = (hi - lo + kGatherTileRows - 1) / kGatherTileRows;
  uint32_t parity = 0u;  // bit b: phase parity to wait for on buffer b

  // pass 0: step-1 rows of early items; pass 1: the rest (after the wait);
  // pass 2: plain gather, every row from its location.
  // Stage 1: the lane's entry (selected row or location) of local chunk li.
  auto load_entry = [&](int li, int pass) -> uint32_t {
    const int g = lo + li * kGatherTileRows + lane;
    if (li >= n_local || g >= hi) return 0u;
    const GatherItem& it = P.items[find_item_entry(P, g)];
    const int e = g - it.ent0;
    if (pass == 0) return (c.early && it.sel) ? (uint32_t)it.sel[e] : 0u;
    if (pass == 1 && !((s_mask[li] >> lane) & 1u)) return 0u;
    return it.loc[e];
  };
  // Stage 2: the lane's row address for local chunk li from its entry.
  auto prep = [&](int li, int pass, uint32_t entry) -> TmaSlot {
    TmaSlot t{nullptr, nullptr, false, 0u};
    if (li >= n_local) return t;
    const int g = lo + li * kGatherTileRows + lane;
    const bool valid = g < hi;
    const GatherItem& it = P.items[find_item_entry(P, valid ? g : hi - 1)];
    t.dst = it.staging + (size_t)(g - it.ent0) * rb;
    if (pass == 0) {
      const bool early = c.early && it.sel != nullptr;
      const uint8_t* p = (early && valid) ? step1_ptr(c, it, (int32_t)entry) : nullptr;
      const unsigned defer = __ballot_sync(0xFFFFFFFFu, valid && p == nullptr);
      if (lane == 0) s_mask[li] = defer;
      t.src = p;
      t.mine = p != nullptr;
    } else {
      t.mine = pass == 2 ? valid : ((s_mask[li] >> lane) & 1u) != 0u;
      if (t.mine) t.src = row_ptr(c, entry);
    }
    return t;
  };
  auto issue = [&](TmaSlot& t, int b) {
    uint8_t* row = s_dyn + b * buf_bytes + (size_t)lane * rb;
    const bool load = t.mine && t.src != nullptr;
    if (t.mine && !load) {  // zeros: plain stores, then hand over to the async proxy
      for (uint32_t o = 0; o < rb; o += 16)
        *reinterpret_cast<uint4*>(row + o) = make_uint4(0u, 0u, 0u, 0u);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    t.lmask = __ballot_sync(0xFFFFFFFFu, load);
    if (t.lmask) {
      if (lane == 0) mbar_arrive_expect(&s_bar[b], (uint32_t)__popc(t.lmask) * rb);
      __syncwarp();
      if (load) bulk_load(row, t.src, rb, &s_bar[b]);
    }
  };
  auto drain = [&](const TmaSlot& t, int b) -> bool {
    if (t.lmask) {
      if (!mbar_wait(&s_bar[b], (parity >> b) & 1u)) {
        if (lane == 0) atomicOr(c.status, kStatusEtimeout);
        return false;
      }
      parity ^= 1u << b;
    }
    __syncwarp();
    if (t.mine)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                   ::"l"(t.dst), "r"(smem_u32(s_dyn + b * buf_bytes + (size_t)lane * rb)),
                     "r"(rb)
                   : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");  // one group per chunk
    return true;
  };
  auto run_pass = [&](int pass) -> bool {
    if (n_local == 0) return true;
    uint32_t e1 = load_entry(1, pass), e2 = load_entry(2, pass), e3 = 0u;
    TmaSlot cur = prep(0, pass, load_entry(0, pass));
    issue(cur, 0);
    TmaSlot nxt = prep(1, pass, e1);
    for (int li = 0; li < n_local; ++li) {
      const int b = li & 1;
      e3 = load_entry(li + 3, pass);  // in flight while chunk li drains
      if (li + 1 < n_local) {
        // the other buffer last held chunk li-1: its stores must have read it
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        issue(nxt, b ^ 1);
      }
      const TmaSlot after = prep(li + 2, pass, e2);
      if (!drain(cur, b)) return false;
      cur = nxt;
      nxt = after;
      e2 = e3;
    }
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    return true;
  };

  if (c.early) {
    if (run_pass(0)) {
      __syncwarp();
      unsigned any = 0u;
      for (int li = lane; li < n_local; li += 32) any |= s_mask[li];
      if (__any_sync(0xFFFFFFFFu, any != 0u)) {
        // rows that needed the hot cache: wait for the resolve / host-copy grids
        asm volatile("griddepcontrol.wait;" ::: "memory");
        run_pass(1);
      }
    }
  } else {
    // locations come from the resolve grid when this launch overlaps it
    // (a no-op without programmatic dependent launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    run_pass(2);
  }
  // staging writes complete (not only their shared-memory reads) before the
  // grid-level ticket
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  finish_grid(P);
}

template <int MAXI>
cudaError_t launch_t(const GatherCommon& c, const GatherItem* items, int n,
                     bool pdl, int impl, cudaStream_t stream) {
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
  if (impl == 1) {
    // persistent grid: as many warps as fit, each with at most kTmaMaxLocal
    // chunks of 32 entries
    int grid = c.tma_grid;
    const int64_t per_warp = kTmaMaxLocal * (int64_t)kGatherTileRows;
    if ((int64_t)grid * per_warp < c.n_entries) grid = (int)((c.n_entries + per_warp - 1) / per_warp);
    if (grid > c.n_tiles) grid = c.n_tiles;
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kTmaThreads);
    cfg.dynamicSmemBytes = tma_smem_bytes(c.row_bytes);
    return cudaLaunchKernelEx(&cfg, gather_tma_kernel<MAXI>, P);
  }
  cfg.blockDim = dim3(kGatherThreads);
  if (c.row_bytes == 1152) return cudaLaunchKernelEx(&cfg, gather_kernel<MAXI, 72>, P);
  return cudaLaunchKernelEx(&cfg, gather_kernel<MAXI, 0>, P);
}

cudaError_t tma_smem_limit(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(gather_tma_kernel<kGatherItemsSmall>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gather_tma_kernel<kGatherItemsLarge>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t gather_set_carveout() {
  const void* ks[] = {
      (const void*)gather_kernel<kGatherItemsSmall, 72>, (const void*)gather_kernel<kGatherItemsSmall, 0>,
      (const void*)gather_kernel<kGatherItemsLarge, 72>, (const void*)gather_kernel<kGatherItemsLarge, 0>,
      (const void*)gather_tma_kernel<kGatherItemsSmall>, (const void*)gather_tma_kernel<kGatherItemsLarge>};
  for (const void* k : ks) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
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


namespace dhs {

int gather_tma_grid(int row_bytes) {
  int dev = 0, sms = 0, per_sm = 0;
  const size_t smem = tma_smem_bytes(row_bytes);
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (tma_smem_limit(smem) != cudaSuccess) return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gather_tma_kernel<kGatherItemsLarge>,
                                                    kTmaThreads, smem) != cudaSuccess)
    return 0;
  return per_sm > 0 ? sms * per_sm : 0;
}

}  // namespace dhs
