// Gather kernel: staging[item][q][i] = the KV row at loc[item][q][i].
//
// "Adaptive DHiSparse", How it works: selected rows are consumed by sparse
// attention from verification staging; Reuse layers gather an inherited
// location vector.  This is the byte-dominant step of the decode path (2 x
// 1152 bytes per entry against 4 bytes of location), a pure HBM copy, so it
// is built for coalescing, not arithmetic:
//   * one CTA per tile of 32 entries of one item; the 32 locations are
//     decoded once into shared memory (tier -> arena, bounds-checked);
//   * the tile is 32 x 72 chunks of 16 bytes = 2304 chunks = 9 per thread;
//     consecutive threads read consecutive 16-byte chunks of a row (each
//     1152-byte row is nine whole 128-byte lines) and write consecutive
//     chunks of the contiguous staging tile, so every load and store is a
//     full-line coalesced access;
//   * all nine loads are issued before the first store (36 KB in flight per
//     CTA) to cover HBM latency; loads use the non-coherent no-allocate path.
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

// CPR = 16-byte chunks per row (0: runtime value).
template <int MAXI, int CPR>
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(const __grid_constant__ GatherParams<MAXI> P) {
  __shared__ const uint8_t* s_src[kGatherTileRows];
  const GatherCommon& c = P.c;
  const int tile = blockIdx.x;
  const GatherItem& it = P.items[find_item(P, tile)];
  const int e0 = (tile - it.tile0) * kGatherTileRows;
  const int ne = min(kGatherTileRows, it.n - e0);
  const int tid = threadIdx.x;
  if (tid < ne) s_src[tid] = row_ptr(c, it.loc[e0 + tid]);
  __syncthreads();
  const int cpr = CPR ? CPR : (c.row_bytes >> 4);
  uint8_t* dst = it.staging + (size_t)e0 * c.row_bytes;
  const int total = ne * cpr;
  if constexpr (CPR != 0) {
    constexpr int U = (kGatherTileRows * CPR + kGatherThreads - 1) / kGatherThreads;
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = tid + u * kGatherThreads;
      if (ch < total) {
        const int e = ch / CPR, p = ch - e * CPR;
        const uint8_t* s = s_src[e];
        v[u] = s ? ld_stream(s + p * 16) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = tid + u * kGatherThreads;
      if (ch < total) *reinterpret_cast<uint4*>(dst + (size_t)ch * 16) = v[u];
    }
  } else {
    for (int ch = tid; ch < total; ch += kGatherThreads) {
      const int e = ch / cpr, p = ch - e * cpr;
      const uint8_t* s = s_src[e];
      const uint4 v = s ? ld_stream(s + p * 16) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dst + (size_t)ch * 16) = v;
    }
  }
}

template <int MAXI>
cudaError_t launch_t(const GatherCommon& c, const GatherItem* items, int n,
                     cudaStream_t stream) {
  GatherParams<MAXI> P;
  P.c = c;
  P.c.n_items = n;
  for (int i = 0; i < n; ++i) P.items[i] = items[i];
  if (c.n_tiles <= 0) return cudaSuccess;
  if (c.row_bytes == 1152)
    gather_kernel<MAXI, 72><<<c.n_tiles, kGatherThreads, 0, stream>>>(P);
  else
    gather_kernel<MAXI, 0><<<c.n_tiles, kGatherThreads, 0, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather(const GatherCommon& c, const GatherItem* items, int n_items,
                          int impl, cudaStream_t stream) {
  (void)impl;
  if (n_items <= 0) return cudaSuccess;
  if (n_items <= kGatherItemsSmall) return launch_t<kGatherItemsSmall>(c, items, n_items, stream);
  if (n_items <= kGatherItemsLarge) return launch_t<kGatherItemsLarge>(c, items, n_items, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dhs
