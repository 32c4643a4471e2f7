// cache_common.cuh -- layout of the cache manager's device scratch and the claim
// step of the guaranteed recall, shared by the cache-manager kernel and by the
// top-k kernel (which performs the claims for the selection it writes).
//
// Claim (ECHO review, marsggbo.github.io, "OSDI'26 | ECHO", section 5.2 "Recall":
// look up HostTokenToGPU for the selected host rows, inf = missing): selected
// entry f of request b, token p, maps to host row h = req_to_host[b][p].  A
// resident row is a hit: its priority becomes the step clock (the "protect" of
// section 5.2 "Free") and the entry competes in slot_claim[slot] with atomicMin.
// A missing row is claimed in HostTokenToGPU with atomicMin(kClaim + f).  Either
// way the lowest entry index -- the first occurrence in (b, j, i) order -- owns
// the row, whatever order the atomics land in.
#pragma once

#include "echo_common.cuh"

namespace echo {

constexpr int kHistBins = 4096;
// Score histograms the decode step's indexer fills for its top-k: one per score row
// (request, query) for the first kSelHintRows rows, kSelBins bins over a window of
// the order-preserving score keys predicted from the row's previous step
constexpr int kSelBins = 2048;
constexpr int kSelBinBits = 11;
constexpr int kSelHintRows = 64;
constexpr int kHistLevels = 4;  // level 0 by age (12 bits); refinements of 12, 12, 8 bits
constexpr int kMaxGrid = 1024;

// global scratch counters (zero between calls)
// kGBar / kGGen: the grid barrier's arrival count and generation
enum { kGValid = 0, kGHits, kGBar, kGRepeats, kGFilled, kGGen, kGCount = 16 };
// per-CTA counts
enum { kCOwn = 0, kCLt, kCEq, kCFree, kCVals };
// ws.ctr: results readable after a call
enum { kCtrMisses = 0, kCtrGranted = 1, kCtrCount = 16 };

struct Workspace {
  int32_t *slot_claim;  // [n_g]  lowest entry index of this step's hits (INT32_MAX = none)
  int32_t *entry_rows;  // [max_rows] host row per entry (append)
  int32_t *entry_h;     // [max_rows] host row of every entry, -1 if none
  int32_t *ent_aux;     // [max_rows] after a claim: HostTokenToGPU as the claim saw it; after the
                        // classification: >= 0 hit slot, -1 none, -2 owned miss, -3 - f1 repeat of f1
  int32_t *miss_f;      // [max_rows] entry index of the r-th owned miss
  int32_t *miss_h;      // [max_rows] host row of the r-th owned miss
  int32_t *miss_rank;   // [max_rows] by entry: rank of an owned miss
  int32_t *miss_stage;  // [max_rows] by entry: staging row index, -1 = not staged
  int32_t *miss_src;    // [max_rows] staging row index of the r-th owned miss, -1 = host pool
  int32_t *alloc_slot;  // [max_rows] the r-th free slot (taken by the r-th miss)
  uint32_t *hist;       // [kHistLevels][kHistBins]
  uint32_t *cta;        // [kMaxGrid][kCVals]
  uint32_t *glob;       // [kGCount]
  int32_t *ctr;         // [kCtrCount]
  uint32_t *sel_hist;   // [kSelHintRows][kSelBins] scores per key bin (zero between steps)
  int4 *sel_hint;       // [kSelHintRows] window of each row's bins: {low key, shift, valid, 0}
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t ws_layout(int32_t n_g, int32_t max_rows, uintptr_t base, Workspace *w) {
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off += ws_align(n * sizeof(int32_t));
    return base + o;
  };
  const size_t R = static_cast<size_t>(max_rows);
  Workspace x;
  x.slot_claim = reinterpret_cast<int32_t *>(take(static_cast<size_t>(n_g)));
  x.entry_rows = reinterpret_cast<int32_t *>(take(R));
  x.entry_h = reinterpret_cast<int32_t *>(take(R));
  x.ent_aux = reinterpret_cast<int32_t *>(take(R));
  x.miss_f = reinterpret_cast<int32_t *>(take(R));
  x.miss_h = reinterpret_cast<int32_t *>(take(R));
  x.miss_rank = reinterpret_cast<int32_t *>(take(R));
  x.miss_stage = reinterpret_cast<int32_t *>(take(R));
  x.miss_src = reinterpret_cast<int32_t *>(take(R));
  x.alloc_slot = reinterpret_cast<int32_t *>(take(R));
  x.hist = reinterpret_cast<uint32_t *>(take(static_cast<size_t>(kHistLevels) * kHistBins));
  x.cta = reinterpret_cast<uint32_t *>(take(static_cast<size_t>(kMaxGrid) * kCVals));
  x.glob = reinterpret_cast<uint32_t *>(take(kGCount));
  x.ctr = reinterpret_cast<int32_t *>(take(kCtrCount));
  x.sel_hist = reinterpret_cast<uint32_t *>(take(static_cast<size_t>(kSelHintRows) * kSelBins));
  x.sel_hint = reinterpret_cast<int4 *>(take(static_cast<size_t>(kSelHintRows) * 4));
  if (w) *w = x;
  return off;
}

struct PoolView {
  uint8_t *free_;
  int32_t *prio, *idxbuf, *to_host, *h2g, *counters;
  uint16_t *gpu_kv;
  const uint16_t *host_kv;
  int32_t n_g, n_h;
  int32_t row_chunks;  // 16-byte pieces of a row (72 for MLA's latent row)
};

// What the top-k kernel needs to claim the entries it selects.
struct ClaimArgs {
  PoolView pool;
  Workspace ws;
  const int32_t *req_to_host;  // [B][L_max]
  int32_t clock;
  const int32_t *clock_dev;
  int32_t *status;
};

// Claim of entry f (token p of request b); h = -1 for padding.  Records the
// entry's host row in ws.entry_h.
// Bin of score key `key` in a row's histogram window {lo, shift}: -1 below the
// window, the last bin for every key above it (so the bins stay ordered like the keys)
__device__ __forceinline__ int sel_bin(uint32_t key, uint32_t lo, uint32_t shift) {
  if (key < lo) return -1;
  const uint32_t b = (key - lo) >> shift;
  return b < static_cast<uint32_t>(kSelBins) ? static_cast<int>(b) : kSelBins - 1;
}

__device__ __forceinline__ void claim_entry(const PoolView &pool, const Workspace &ws, int f, int32_t h,
                                            int32_t clock, int32_t *status) {
  if (h >= pool.n_h) {
    set_status(status, ECHO_DEV_BAD_INDEX);
    h = -1;
  }
  if (h < 0) {
    ws.entry_h[f] = -1;
    return;
  }
  const int32_t v = pool.h2g[h];
  if (v >= 0 && v < pool.n_g) {
    pool.prio[v] = clock;              // protect + LRU clock
    red_min(ws.slot_claim + v, f);   // the first entry of the row owns the hit
  } else if (v == kInf || v < 0) {
    red_min(pool.h2g + h, kClaim + f);  // the first entry of the row owns the miss
  } else {
    set_status(status, ECHO_DEV_BAD_INDEX);
    h = -1;
  }
  ws.entry_h[f] = h;
  ws.ent_aux[f] = v;  // the map entry seen here: a hit's slot stays valid for the step
}

}  // namespace echo
