// Internal launch interface between the host pool manager (pool.cpp) and
// the sm_103a kernels (resolve.cu, hostcopy.cu, gather.cu, append.cu).
// Not part of the C ABI.
//
// Item tables travel by value in the kernel parameter space
// (__grid_constant__), so a decode step needs no host-to-device copy of its
// descriptors and stays capturable as plain kernel launches.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dhs {

constexpr uint32_t kTierTail = 0u, kTierOpt = 1u, kTierHot = 2u;
constexpr uint32_t kNoLoc = 0xFFFFFFFFu;
constexpr uint32_t kEndLoc = 0xFFFFFFFEu;  // past the end of a union location list
constexpr uint32_t kStatusErange = 1u, kStatusEbudget = 2u, kStatusEloc = 4u;
constexpr uint32_t kStatusEtimeout = 8u;
constexpr int32_t kErrRange = -5, kErrBudget = -4;  // DHS_ERANGE, DHS_EBUDGET
constexpr int kMaxHotRows = 16384;

// Polls for a published loc_ready / copy_ready mark before falling back to
// waiting for the grids (DHS_OPT_MARK_POLLS default).
constexpr uint32_t kMarkPolls = 1u << 20;

// Sequence numbers of resolve launches as published in loc_ready / copy_ready
// marks (never 0, which is what a zeroed mark holds).
constexpr uint32_t kSeqMask = 0x1FFFFFFFu;
// copy_ready mark bit: the item has no misses, so its copy reads nothing of it
constexpr uint32_t kMarkNoMiss = 0x20000000u;
// copy_ready mark bit: the miss count and lists are written, the staging
// entries not yet (a second store clears the bit once they are)
constexpr uint32_t kMarkEntriesPending = 0x40000000u;

// Optional timeline (DHS_OPT_TRACE): per kernel kind, the earliest CTA start
// and the latest CTA end in %globaltimer nanoseconds.
enum TraceSlot { kTraceResolve = 0, kTraceCopy = 1, kTraceGather = 2, kTraceLater = 3,
                 kTraceKinds = 4 };

// Fused steps: rows in hot slots that this step's host copy fills ("fresh"
// rows) are the only ones a gather must leave until the copy grid is done.
// Gather tiles append them to a device list of LaterEntry, copied by a
// second launch once the copy grid has completed.
struct LaterEntry {
  uint8_t* dst;   // staging row (null: unused slot)
  uint32_t loc;   // hot location of the row
  uint32_t pad;
};

#ifdef __CUDACC__
__device__ __forceinline__ unsigned long long trace_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Called by thread 0 of every CTA at start (end = false) and at end.
__device__ __forceinline__ void trace_mark(unsigned long long* trace, int kind, bool end) {
  if (!trace) return;
  const unsigned long long t = trace_now();
  if (end) atomicMax(&trace[2 * kind + 1], t);
  else atomicMin(&trace[2 * kind], t);
}
#endif

// ------------------------------------------------------------ resolve (a-c)
constexpr int kResolveItemsLarge = 256, kResolveItemsSmall = 32;
// Threads per resolve CTA (a whole CTA per item).  A launch of at most
// kResolveItemsSmall items leaves most SMs to the gather that overlaps it,
// and its CTAs share their SMs with that gather: 512 threads there.  Larger
// launches fill the GPU, and each item's copy starts when it is resolved:
// 1024 threads there.
constexpr int resolve_threads(int max_items) {
  return max_items <= kResolveItemsSmall ? 512 : 1024;
}
// A large launch whose shared-memory plan lets two CTAs share an SM can run
// 512-thread CTAs two per SM instead: more items than SMs then resolve in one
// wave instead of two.
constexpr int kResolvePairThreads = 512;

struct ResolveItem {
  const int32_t* sel;   // [n] selected rows (Q*k, verify queries back to back)
  uint32_t* loc;        // [n] locations out
  uint32_t* counters;   // [8] or null
  int64_t L;            // current length (after this step's append)
  int64_t N;            // imported rows
  int32_t pair;         // req * S + src
  int32_t n;            // Q * k
  // decode rows appended by this launch (dhs_decode_step), else count 0
  const uint8_t* app_rows;  // [app_count][row_bytes] device
  uint8_t* app_host;        // device-visible pointer of the pair's host rows
                            // (null: a window source, no host copy)
  int64_t app_L0;           // length before the append
  int32_t app_count;
  int16_t stage;       // list, per miss, the entries that selected it (host
                       // copy writes them into staging)
  int16_t loc_shared;  // a gather-only item of the launch reads `loc` too
  int32_t* index;  // union staging: [n] union rank of each entry; null = per-query
  int64_t lo;      // lowest row the source serves: 0, or L - T for a window source
};

struct ResolveCommon {
  int32_t* tags;         // [pairs][B]
  uint32_t* stamps;      // [pairs][B]
  const int32_t* map;    // [pairs][Pmax]
  int32_t* miss_rows;    // [pairs][Mcap]
  int32_t* miss_slots;   // [pairs][Mcap]
  uint32_t* miss_count;  // [pairs]
  uint32_t* copy_cursor; // [pairs] miss rows the host copy has claimed (zeroed here)
  int32_t* pair_status;  // [pairs]
  uint32_t* status;      // sticky flags
  int32_t T, B, Pmax, Mcap;
  int32_t page_shift;    // log2(page_rows)
  int32_t w64cap;        // bitmap words reserved in shared memory
  int32_t qkcap;         // candidate slots reserved in shared memory
  uint32_t step;
  int32_t n_items;
  int32_t row_bytes;
  uint8_t* tail;         // tail arena (appends folded into the launch)
  unsigned long long* trace;  // null = off
  uint32_t seq;          // sequence number of this launch
  int32_t uni;           // shared-memory plan includes the union bitmap
  uint32_t* loc_ready;   // [pairs] seq once the item's locations are written; null = off
  uint32_t* copy_ready;  // [pairs] seq once its miss lists (and staging entries) are written
  uint32_t* fill;        // [pairs][fill_words] hot slots filled by this step's copy
  uint32_t* later_count; // [2] fresh-row list lengths; the launch zeroes [gen ^ 1]
  int32_t fill_words;
  uint32_t gen;          // fused-step generation (parity picks the list counter)
  int32_t* miss_off;     // [pairs][Mcap + 1] per miss: first entry in miss_ent
  int32_t* miss_ent;     // [pairs][ent_cap] staging entries of the misses
  int32_t ent_cap;
  int32_t selcap;        // selection entries staged in shared memory (0 = none)
};

// Shared-memory plan of one resolve CTA: bitmaps of w64cap words, qkcap
// candidate rows (at most B: more fail the budget before they are listed), B
// slots, and selcap staged selection entries.
size_t resolve_smem_bytes(int w64cap, int qkcap, int B, bool uni, int selcap);
cudaError_t resolve_set_smem_limit(size_t bytes);
// paired: a launch of more than kResolveItemsSmall items as 512-thread CTAs
// two per SM (the caller checks that two plans fit one SM).  ctas: CTAs of
// the grid when below n_items (each then resolves several items in turn),
// else one per item.
cudaError_t launch_resolve(const ResolveCommon& c, const ResolveItem* items,
                           int n_items, int ctas, size_t smem, bool paired,
                           cudaStream_t stream);

// ------------------------------------------------------------ page moves
// Whole optional pages between the optional arena and the pinned host copy
// (refill and admission host -> device, deferred backup device -> host), as
// one launch over a list of pages instead of one copy call per page.
struct PageMove {
  const uint8_t* src;  // device-visible addresses (mapped host or device)
  uint8_t* dst;
};
constexpr int kPageMovesMax = 1024;  // per launch (kernel parameter space)
constexpr int kPageMoveThreads = 512;
cudaError_t launch_page_moves(const PageMove* moves, int n, int page_bytes, int ctas,
                              cudaStream_t stream);

// ------------------------------------------------------------ host copy (d)
constexpr int kCopyThreads = 512;
constexpr int kCopyItemsMax = 256;
constexpr int kCopyItemsSmall = 32;  // a smaller parameter table for small steps

// Gather-only (Reuse) items handed an item's location vector whose staging
// the host copy also writes, per item; further ones take the fresh-row list.
constexpr int kCopyShareMax = 3;

struct CopyItem {
  const uint8_t* host;  // device-visible pointer of the pair's pinned host rows
  uint8_t* staging;     // also write each miss row to its staging entries; null = no
  int32_t pair;
  int32_t nshare;       // staging buffers of gather-only items sharing the locations
  uint8_t* share[kCopyShareMax];  // (the same entries, the same row layout)
};

struct CopyCommon {
  uint8_t* hot;
  const int32_t* miss_rows;
  const int32_t* miss_slots;
  const uint32_t* miss_count;
  uint32_t* cursor;           // [pairs] miss rows claimed so far (the resolve launch zeroes it)
  int32_t B, Mcap, row_bytes, n_items;
  unsigned long long* trace;  // null = off
  const uint32_t* ready;      // [pairs] the resolve launch's copy_ready marks, null = none
  uint32_t seq;               // that launch's sequence number
  int32_t ent_cap;
  const int32_t* miss_off;    // [pairs][Mcap + 1] (items with staging)
  const int32_t* miss_ent;    // [pairs][ent_cap]
  uint32_t mark_polls;        // polls of a copy_ready mark before waiting for the grid;
                              // 0: never read the marks
  int32_t steal;              // 1: rows claimed through the cursors, and blocks done with
                              // their own items take other items' unclaimed rows
};

// threads: per block, a multiple of 32 up to kCopyThreads.  hold_smem:
// dynamic shared memory each block reserves (and leaves unused) so that no
// other CTA shares its SM; at most the limit set by hostcopy_set_carveout.
cudaError_t launch_hostcopy(const CopyCommon& c, const CopyItem* items,
                            int n_items, int ctas, int threads, bool pdl, size_t hold_smem,
                            cudaStream_t stream);

// ------------------------------------------------------------ gather (e)
constexpr int kGatherThreads = 256;
constexpr int kGatherVector = 0, kGatherTma = 1;  // DHS_OPT_GATHER_IMPL values
constexpr int kGatherTileRows = 32;  // entries per tile of the vector gather
// TMA gather tile: kTmaWarps warps per CTA, each moving kTmaWarpRows entries
// under its own mbarrier (lanes past them idle).  A warp's bulk stores wait
// only for its own rows, not for the slowest row of the whole tile.
constexpr int kTmaWarpRows = 8;
constexpr int kTmaWarps = 2;
constexpr int kTmaTileRows = kTmaWarpRows * kTmaWarps;
constexpr int gather_tile_rows(int impl) {
  return impl == kGatherTma ? kTmaTileRows : kGatherTileRows;
}
constexpr int kLaterThreads = 512;
constexpr int kGatherItemsLarge = 384, kGatherItemsSmall = 64;

struct GatherItem {
  const uint32_t* loc;
  uint8_t* staging;
  const int32_t* sel;  // non-null: a resolved item whose step-1 rows may be copied early
  int64_t L, N;        // length and imported rows of the item's source
  int64_t L0;          // rows >= L0 were appended by this launch
  const uint8_t* app;  // their bytes ([L - L0][row_bytes], the append's source), or
                       // null: rows >= L0 are then never early
  int32_t n;           // entries
  int32_t tile0;       // first tile of this item in the launch
  int32_t pair;        // req * S + src (resolved items)
  uint32_t seq;        // sequence number of the resolve launch that resolved it
  uint32_t flags;      // kGiLocReady
};
// The item's locations are those of a pair resolved by the preceding resolve
// launch of the same fused step, published through loc_ready[pair] == seq.
constexpr uint32_t kGiLocReady = 1u;
// The host copy writes the item's fresh rows into its staging itself.
constexpr uint32_t kGiStaged = 2u;

struct GatherCommon {
  const uint8_t* tail;
  const uint8_t* opt;
  const uint8_t* hot;
  const int32_t* map;          // [pairs][Pmax] page map (early phase)
  uint32_t tail_rows, opt_rows, hot_rows;  // arena sizes in rows
  int32_t row_bytes;
  uint32_t* status;
  int32_t n_items;
  int32_t n_tiles;
  int32_t item_tiles;         // tiles of every item when all items have as many, else 0
  int32_t T, Pmax, page_shift;
  int32_t early;             // copy step-1 rows before waiting for the resolve grid
  unsigned long long* trace;  // null = off
  const uint32_t* loc_ready;  // [pairs] (kGiLocReady items)
  const uint32_t* fill;       // [pairs][fill_words]
  int32_t fill_words;
  int32_t B;
  LaterEntry* later;          // fresh-row list, null = fresh rows wait in their tile
  uint32_t* later_count;      // [2]
  uint32_t later_cap;
  uint32_t gen;
  int32_t tpc;                // TMA gather: consecutive tiles per CTA (>= 1)
  int32_t read_once;          // no row of the launch is read twice (one query per item,
                              // no gather-only item): bulk loads hint L2 evict-first
  uint32_t mark_polls;        // polls of a loc_ready mark before waiting for the grids
};

// Each kernel file sets its kernels' shared-memory carveout to the maximum,
// so consecutive kernels of a step never make an SM reconfigure its L1 /
// shared split.
cudaError_t resolve_set_carveout();
cudaError_t hostcopy_set_carveout(size_t hold_smem);
cudaError_t gather_set_carveout();
cudaError_t append_set_carveout();

cudaError_t launch_gather(const GatherCommon& c, const GatherItem* items,
                          int n_items, bool pdl, int impl, cudaStream_t stream);
// Copy the fresh-row list of generation c.gen once the gather (and through
// it the copy grid) has completed; programmatic dependent of the gather.
cudaError_t launch_gather_later(const GatherCommon& c, int ctas, cudaStream_t stream);

// Raise the TMA gather's dynamic shared-memory limit for a row size.
// *tma_ok: whether the TMA gather's 16-row tile of this row size fits in
// `optin` bytes of shared memory per block (else only the vector gather runs).
cudaError_t gather_set_smem_limit(int row_bytes, int optin, bool* tma_ok);

// ------------------------------------------------------------ append (A0)
constexpr int kAppendThreads = 256;
constexpr int kAppendItemsMax = 256;

struct AppendItem {
  const uint8_t* rows;  // [count][row_bytes] device
  uint8_t* host;        // device-visible pointer of the pair's host rows (null: a
                        // window source, whose rows go to the tail ring only)
  int64_t L0;           // length before the append
  int32_t pair;
  int32_t count;
};

struct AppendCommon {
  uint8_t* tail;
  int32_t T, row_bytes, n_items, pad;
};

cudaError_t launch_append(const AppendCommon& c, const AppendItem* items,
                          int n_items, cudaStream_t stream);

}  // namespace dhs

namespace dhs {

// ------------------------------------------------------------ no-alloc scratch
// Fixed miss-list storage for dhs_resolve_noalloc (noalloc_scratch.cu):
// up to kNoallocMissCap (row, slot) entries, i.e. pairs * min(B, Q*k) of the
// pool, and kNoallocPairs per-pair counts.
constexpr int kNoallocMissCap = 65536;
constexpr int kNoallocPairs = 4096;
constexpr int kNoallocMaxDevices = 64;

struct NoallocScratch {
  int32_t* miss_rows;
  int32_t* miss_slots;
  uint32_t* miss_count;
};

// Device address of the scratch on the current device (looked up once per
// device with cudaGetSymbolAddress).
cudaError_t noalloc_scratch(NoallocScratch* out);

}  // namespace dhs
