// Fixed device-side scratch for dhs_resolve_noalloc.
//
// dhs_resolve keeps its per-item miss lists (the rows step 3 must fetch and
// the hot slots they go to) in the caller-allocated metadata buffer.  Some
// callers cannot allocate device memory at the point where they resolve --
// for example an embedding runtime that hands the library only the buffers
// it owns, or code that runs where allocation calls are not permitted -- so
// dhs_resolve_noalloc puts those lists in this file-scope array instead.
// The array lives in the library image: every GPU that loads libdhs.so
// holds it (540,672 bytes) until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// is only a stand-in symbol), so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, the first
// time the entry point runs there.
#include <mutex>

#include "dhs_internal.h"

namespace dhs {

// [0, kNoallocMissCap): miss rows; [kNoallocMissCap, 2*kNoallocMissCap):
// miss slots; then kNoallocPairs miss counts.
static __device__ __align__(256) int32_t g_noalloc_scratch[2 * kNoallocMissCap + kNoallocPairs];

namespace {
std::mutex g_mu;
void* g_addr[kNoallocMaxDevices] = {nullptr};
}  // namespace

cudaError_t noalloc_scratch(NoallocScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_addr[dev] = p;
  }
  int32_t* base = static_cast<int32_t*>(g_addr[dev]);
  out->miss_rows = base;
  out->miss_slots = base + kNoallocMissCap;
  out->miss_count = reinterpret_cast<uint32_t*>(base + 2 * kNoallocMissCap);
  return cudaSuccess;
}

}  // namespace dhs
