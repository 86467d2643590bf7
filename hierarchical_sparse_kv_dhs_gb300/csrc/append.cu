// Append kernel: decode rows enter the mutable tail ring and are written
// through to the pinned host copy.
//
// "Adaptive DHiSparse", How it works / Memory split (a mutable tail per
// request and KV source) and Reclamation and refill (no row is left without
// a copy: it is ready on the GPU or backed on the host); Limits (decode rows
// are served the hot-cache way), so once a decode row leaves the tail it is
// found only through the hot cache or the host copy.  Row L+j of
// a pair goes to tail slot (L+j) mod T and to host row L+j.  A window source
// ("Speculative state": a drafter retains only the rows its window covers,
// stored as a ring) has no host copy: its rows go to the ring only.
#include "dhs_internal.h"

namespace dhs {
namespace {

template <int MAXI>
struct AppendParams {
  AppendCommon c;
  AppendItem items[MAXI];
};
// kernel parameter space holds at most 32764 bytes
static_assert(sizeof(AppendParams<kAppendItemsMax>) <= 32764, "append item table too large");

template <int MAXI>
__global__ void __launch_bounds__(kAppendThreads)
    append_kernel(const __grid_constant__ AppendParams<MAXI> P) {
  const AppendCommon& c = P.c;
  const AppendItem& it = P.items[blockIdx.x];
  const int rb = c.row_bytes, cpr = rb >> 4;
  const int total = it.count * cpr;
  for (int ch = threadIdx.x; ch < total; ch += blockDim.x) {
    const int j = ch / cpr, p = ch - j * cpr;
    const int64_t row = it.L0 + j;
    const uint4 v = *reinterpret_cast<const uint4*>(it.rows + (size_t)j * rb + p * 16);
    uint8_t* t = c.tail + ((size_t)it.pair * c.T + (size_t)(row % c.T)) * rb + p * 16;
    *reinterpret_cast<uint4*>(t) = v;
    if (it.host) *reinterpret_cast<uint4*>(it.host + (size_t)row * rb + p * 16) = v;
  }
}

}  // namespace

cudaError_t append_set_carveout() {
  return cudaFuncSetAttribute(append_kernel<kAppendItemsMax>, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
}

cudaError_t launch_append(const AppendCommon& c, const AppendItem* items, int n_items,
                          cudaStream_t stream) {
  if (n_items <= 0) return cudaSuccess;
  if (n_items > kAppendItemsMax) return cudaErrorInvalidValue;
  AppendParams<kAppendItemsMax> P;
  P.c = c;
  P.c.n_items = n_items;
  for (int i = 0; i < n_items; ++i) P.items[i] = items[i];
  append_kernel<kAppendItemsMax><<<n_items, kAppendThreads, 0, stream>>>(P);
  return cudaGetLastError();
}

}  // namespace dhs
