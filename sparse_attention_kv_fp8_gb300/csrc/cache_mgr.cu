// cache_mgr.cu -- the graph-friendly cache manager and the guaranteed recall.
//
// ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"), section 5: fixed-length
// integer metadata on the GPU (GPUTokenFree, GPUTokenPriority, GPUIndicesBuffer,
// GPUTokenToHost, HostTokenToGPU), updated only by parallel device operations so
// that the whole decode step replays from one CUDA graph:
//   Allocate -- free-slot threads take atomic tickets; tickets below the request
//               size win; priority raised; both maps set; indices to the buffer.
//   Free     -- protect the step's selection, arg-top-k of the lowest priorities,
//               scatter; no data moves (the host already holds every row).
//   Recall   -- look up HostTokenToGPU for the selected host rows (inf = missing),
//               free + allocate, set the maps, copy the KV host -> GPU from kernels
//               reading the mapped host memory.
//
// sm_103a design.  Three kernels per operation, all fixed-shape:
//   claim  (grid-wide)  maps each selected entry to its host row; resident rows
//                       are hits (priority = clock, protecting them); missing rows
//                       are claimed in HostTokenToGPU with atomicMin(kClaim + f),
//                       so the first entry in (b, j, i) order owns each row.
//   plan   (one 8-CTA thread-block cluster) compacts the owned misses in entry
//                       order, selects the victims -- the smallest (priority, slot)
//                       by a 3-pass radix select with distributed-shared-memory
//                       histograms -- and hands the lowest free slots to the
//                       misses in order.  Block and cluster prefix scans replace
//                       the page's atomic ticket race with its slot-ordered
//                       interleaving, so the metadata is deterministic.
//   copy   (grid-wide)  moves each recalled row (1152 B, 16-byte vectors, several
//                       rows in flight per warp) from the staging area or the
//                       pinned host pool into its slot and writes out_slot.
#include "cluster_select.cuh"

ECHO_TRACE_UNIT(cache_mgr)

namespace echo {

enum PlanMode { kModeRecall = 0, kModeAlloc = 1, kModeAppend = 2, kModeEvict = 3 };

// workspace counters
enum { kCtrMisses = 0, kCtrGranted = 1, kCtrCount = 16 };

struct Workspace {
  int32_t *slot_claim;  // [n_g]  min entry index protecting the slot (INT32_MAX = none)
  int32_t *entry_rows;  // [max_rows] host row per entry (append)
  int32_t *miss_f;      // [max_rows] entry index of the r-th owned miss
  int32_t *miss_h;      // [max_rows] host row of the r-th owned miss
  int32_t *miss_stage;  // [max_rows] by entry: staging row index, -1 = not staged
  int32_t *alloc_slot;  // [max_rows] slot granted to the r-th miss
  int32_t *ctr;         // [kCtrCount]
};

__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline size_t ws_layout(int32_t n_g, int32_t max_rows, uintptr_t base, Workspace *w) {
  size_t off = 0;
  auto take = [&](size_t n) {
    size_t o = off;
    off += ws_align(n * sizeof(int32_t));
    return reinterpret_cast<int32_t *>(base + o);
  };
  Workspace x;
  x.slot_claim = take(static_cast<size_t>(n_g));
  x.entry_rows = take(static_cast<size_t>(max_rows));
  x.miss_f = take(static_cast<size_t>(max_rows));
  x.miss_h = take(static_cast<size_t>(max_rows));
  x.miss_stage = take(static_cast<size_t>(max_rows));
  x.alloc_slot = take(static_cast<size_t>(max_rows));
  x.ctr = take(kCtrCount);
  if (w) *w = x;
  return off;
}

struct PoolView {
  uint8_t *free_;
  int32_t *prio, *idxbuf, *to_host, *h2g, *counters;
  uint16_t *gpu_kv;
  const uint16_t *host_kv;
  int32_t n_g, n_h;
};

struct PlanParams {
  PoolView pool;
  Workspace ws;
  int mode;
  int F;  // entries
  // recall entries
  const int32_t *sel;
  const int32_t *req_to_host;
  int n_q, k, L_max;
  // alloc / append entries
  const int32_t *rows;
  const int32_t *n_dev;
  int32_t *out_slots;
  // evict
  const int32_t *evict_n_dev;
  // staging (recall)
  const int32_t *stage_host;
  const int32_t *stage_count;
  const int32_t *ctx_len;
  int B, stage_stride, cap_div;
  int32_t clock;
  const int32_t *clock_dev;
  echo_stats *stats;
  int32_t *status;
};

__device__ __forceinline__ int32_t read_clock(const PlanParams &P) { return P.clock_dev ? *P.clock_dev : P.clock; }

// host row of entry f, or -1 (with BAD_INDEX flagged for out-of-range indices)
__device__ __forceinline__ int32_t entry_row(const PlanParams &P, int f, int n_entries, bool flag) {
  if (f >= n_entries) return -1;
  int32_t h;
  if (P.mode == kModeRecall) {
    const int32_t p = P.sel[f];
    if (p < 0) return -1;
    if (p >= P.L_max) {
      if (flag) set_status(P.status, ECHO_DEV_BAD_INDEX);
      return -1;
    }
    h = P.req_to_host[static_cast<size_t>(f / (P.n_q * P.k)) * P.L_max + p];
  } else {
    h = P.rows[f];
    if (h < 0 && P.mode == kModeAppend) return -1;  // request skipped by append
  }
  if (h < 0 || h >= P.pool.n_h) {
    if (flag) set_status(P.status, ECHO_DEV_BAD_INDEX);
    return -1;
  }
  return h;
}

__device__ __forceinline__ int entries_count(const PlanParams &P) {
  if (P.mode == kModeAlloc) {
    int n = *P.n_dev;
    return n < 0 ? 0 : (n > P.F ? P.F : n);
  }
  return P.F;
}

// ---------------------------------------------------------------------------
// claim: hits are protected, misses claim their host row (first entry wins)
// ---------------------------------------------------------------------------
__global__ void claim_kernel(const PlanParams P) {
  const int n = entries_count(P);
  const int32_t clock = read_clock(P);
  for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < n; f += gridDim.x * blockDim.x) {
    const int32_t h = entry_row(P, f, n, true);
    if (h < 0) {
      if (P.mode == kModeAlloc) P.out_slots[f] = -1;
      continue;
    }
    const int32_t v = P.pool.h2g[h];
    const bool resident = v >= 0 && v < P.pool.n_g;
    if (P.mode == kModeRecall) {
      if (resident) {
        P.pool.prio[v] = clock;  // protect + LRU clock
        atomicMin(P.ws.slot_claim + v, f);
      } else if (v == kInf || v < 0) {
        atomicMin(P.pool.h2g + h, kClaim + f);
      } else {
        set_status(P.status, ECHO_DEV_BAD_INDEX);
      }
    } else {
      if (v != kInf && v >= 0) {  // already resident (or corrupt): cannot allocate again
        set_status(P.status, ECHO_DEV_BAD_INDEX);
        if (P.mode == kModeAlloc) P.out_slots[f] = -1;
      } else {
        atomicMin(P.pool.h2g + h, kClaim + f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// plan: one thread-block cluster; every CTA stages its slice of the slots in
// shared memory as one key per slot:
//   kFreeKey          free slot
//   kProtKey          occupied and not evictable (priority >= clock: protected)
//   priority          occupied and evictable
// ---------------------------------------------------------------------------
constexpr uint32_t kFreeKey = 0xFFFFFFFFu;
constexpr uint32_t kProtKey = 0xFFFFFFFEu;
constexpr int kPlanMaxChunk = 48 * 1024;  // slots per CTA (shared memory)

__global__ void __launch_bounds__(kSelThreads, 1) plan_kernel(const PlanParams P) {
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int C = static_cast<int>(cl.num_blocks());
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem *S = reinterpret_cast<SelSmem *>(smem_raw);
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem));
  const int32_t clock = read_clock(P);
  const int n_g = P.pool.n_g;
  const int32_t n_free0 = P.pool.counters[0];
  const int32_t prev_idx = P.pool.counters[1];
  ECHO_TRACE_MARK(0);

  // ===== this CTA's slots, staged =====
  const int sc = (n_g + C - 1) / C;
  const int lo = rank * sc < n_g ? rank * sc : n_g;
  const int hi = lo + sc < n_g ? lo + sc : n_g;
  const int nloc = hi - lo;
  for (int i = threadIdx.x; i < nloc; i += kSelThreads) {
    const int32_t pr = P.pool.prio[lo + i];
    keys[i] = P.pool.free_[lo + i] ? kFreeKey
                                   : ((pr >= 0 && pr < clock) ? static_cast<uint32_t>(pr) : kProtKey);
  }
  __syncthreads();
  // contiguous per-thread segments of the slice, odd length (conflict-free reads)
  int seg = (nloc + kSelThreads - 1) / kSelThreads;
  seg |= 1;
  const int t0 = threadIdx.x * seg < nloc ? threadIdx.x * seg : nloc;
  const int t1 = t0 + seg < nloc ? t0 + seg : nloc;
  ECHO_TRACE_MARK(1);

  // ===== phase A: owned misses in entry order (and unique hits) =====
  uint32_t M = 0, n_sel = 0, n_hit = 0;
  if (P.mode != kModeEvict) {
    const int n = entries_count(P);
    const int c0 = static_cast<int>((static_cast<long long>(n) * rank) / C);
    const int c1 = static_cast<int>((static_cast<long long>(n) * (rank + 1)) / C);
    const int per = (c1 - c0 + kSelThreads - 1) / kSelThreads;
    const int s0 = c0 + threadIdx.x * per < c1 ? c0 + threadIdx.x * per : c1;
    const int s1 = s0 + per < c1 ? s0 + per : c1;
    uint32_t own = 0, hits = 0, valid = 0;
    for (int f = s0; f < s1; ++f) {
      const int32_t h = entry_row(P, f, n, false);
      if (h < 0) continue;
      ++valid;
      const int32_t v = P.pool.h2g[h];
      if (v == kClaim + f) {
        ++own;
      } else if (P.mode == kModeRecall && v >= 0 && v < n_g && P.ws.slot_claim[v] == f) {
        ++hits;
        P.ws.slot_claim[v] = INT32_MAX;  // leave the workspace initialised
      } else if (P.mode != kModeRecall && v < 0) {
        // a repeat of a row an earlier entry claimed: rejected (resident rows were
        // rejected by the claim kernel)
        if (P.mode == kModeAlloc) P.out_slots[f] = -1;
        set_status(P.status, ECHO_DEV_BAD_INDEX);
      }
    }
    uint32_t ex_own, ex_val, t_own, t_val;
    sel_block_scan2(own, valid, ex_own, ex_val, t_own, t_val, S);
    uint32_t pre_own, pre_val, g_own, g_val;
    sel_cluster_prefix2(cl, S, t_own, t_val, pre_own, pre_val, g_own, g_val);
    M = g_own;
    n_sel = g_val;
    uint32_t r = pre_own + ex_own;
    for (int f = s0; f < s1; ++f) {
      const int32_t h = entry_row(P, f, n, false);
      if (h < 0) continue;
      if (P.pool.h2g[h] == kClaim + f) {
        P.ws.miss_f[r] = f;
        P.ws.miss_h[r] = h;
        ++r;
      }
    }
    if (P.mode == kModeRecall) {
      uint32_t eh, dz, th, tz;
      sel_block_scan2(hits, 0, eh, dz, th, tz, S);
      uint32_t ph, pz, gh, gz;
      sel_cluster_prefix2(cl, S, th, 0, ph, pz, gh, gz);
      n_hit = gh;
    }
  }

  ECHO_TRACE_MARK(2);
  // ===== phase A2: which claimed misses the prefetch staged this step =====
  uint32_t staged_total = 0;
  if (P.mode == kModeRecall && P.stage_count != nullptr) {
    const int gw = rank * kSelWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int b = gw; b < P.B; b += C * kSelWarps) {
      int L = P.ctx_len[b];
      L = L < 0 ? 0 : (L > P.L_max ? P.L_max : L);
      int cap = (L + P.cap_div - 1) / P.cap_div;
      cap = cap < P.stage_stride ? cap : P.stage_stride;
      int nb = P.stage_count[b];
      nb = nb < cap ? nb : cap;
      for (int i = lane; i < nb; i += 32) {
        const int32_t h = P.stage_host[static_cast<size_t>(b) * P.stage_stride + i];
        if (h < 0 || h >= P.pool.n_h) continue;
        const int32_t v = P.pool.h2g[h];
        if (v < 0) {
          const uint32_t f = static_cast<uint32_t>(v) - 0x80000000u;  // v = kClaim + f
          if (f < static_cast<uint32_t>(P.F)) P.ws.miss_stage[f] = b * P.stage_stride + i;
        }
      }
      if (lane == 0) staged_total += static_cast<uint32_t>(nb);
    }
  }

  ECHO_TRACE_MARK(3);
  // ===== phase B: evict E slots, the smallest (priority, slot) among evictable ones =====
  int32_t E = 0;
  if (P.mode == kModeEvict) {
    E = *P.evict_n_dev;
    E = E < 0 ? 0 : E;
  } else if (P.mode != kModeAlloc) {
    E = static_cast<int32_t>(M) - n_free0;
    E = E < 0 ? 0 : E;
  }
  if (E > 0) {
    uint32_t cnt = 0, mn = 0xFFFFFFFFu, mx = 0;
    for (int i = t0; i < t1; ++i) {
      const uint32_t key = keys[i];
      if (key < kProtKey) {
        ++cnt;
        mn = min(mn, key);
        mx = max(mx, key);
      }
    }
    uint32_t ec, dz, tc, tz;
    sel_block_scan2(cnt, 0, ec, dz, tc, tz, S);
    uint32_t pc, pz, eligible, gz;
    sel_cluster_prefix2(cl, S, tc, 0, pc, pz, eligible, gz);
    if (static_cast<uint32_t>(E) > eligible) {
      if (rank == 0 && threadIdx.x == 0) set_status(P.status, ECHO_DEV_POOL_EXHAUSTED);
      E = static_cast<int32_t>(eligible);
    }
  }
  if (E > 0) {
    uint32_t mn = 0xFFFFFFFFu, mx = 0;
    for (int i = t0; i < t1; ++i) {
      const uint32_t key = keys[i];
      if (key < kProtKey) {
        mn = min(mn, key);
        mx = max(mx, key);
      }
    }
    ECHO_TRACE_MARK(4);
    uint32_t pmin, pmax;
    sel_cluster_minmax(cl, S, mn, mx, pmin, pmax);
    ECHO_TRACE_MARK(5);
    uint32_t T, needT;
    sel_radix_select(cl, S, nloc, pmin, pmax, static_cast<uint32_t>(E), false,
                     [&](int i, uint32_t &key) {
                       key = keys[i];
                       return key < kProtKey;
                     },
                     T, needT);
    ECHO_TRACE_MARK(6);
    // victims: priority < T, or == T among the first needT in slot order
    uint32_t lt = 0, eq = 0;
    for (int i = t0; i < t1; ++i) {
      const uint32_t key = keys[i];
      lt += key < T;
      eq += key == T;
    }
    uint32_t elt, eeq, tlt, teq;
    sel_block_scan2(lt, eq, elt, eeq, tlt, teq, S);
    uint32_t plt, peq, glt, geq;
    sel_cluster_prefix2(cl, S, tlt, teq, plt, peq, glt, geq);
    uint32_t ob = plt + elt, eb = peq + eeq;
    for (int i = t0; i < t1; ++i) {
      const uint32_t key = keys[i];
      bool victim = false;
      uint32_t pos = 0;
      if (key < T) {
        victim = true;
        pos = ob + (eb < needT ? eb : needT);
        ++ob;
      } else if (key == T) {
        if (eb < needT) {
          victim = true;
          pos = ob + eb;
        }
        ++eb;
      }
      if (!victim) continue;
      const int s = lo + i;
      const int32_t h = P.pool.to_host[s];
      keys[i] = kFreeKey;
      P.pool.free_[s] = 1;
      P.pool.prio[s] = -1;
      if (h >= 0 && h < P.pool.n_h) P.pool.h2g[h] = kInf;
      P.pool.to_host[s] = kInf;
      if (P.mode == kModeEvict) P.pool.idxbuf[pos] = s;
    }
  }
  ECHO_TRACE_MARK(7);
  __syncthreads();
  cl.sync();  // miss lists of every CTA written, evictions done
  ECHO_TRACE_MARK(8);

  // ===== phase C: the r-th miss takes the r-th lowest free slot =====
  int32_t A = 0;
  if (P.mode != kModeEvict) {
    uint32_t nf = 0;
    for (int i = t0; i < t1; ++i) nf += keys[i] == kFreeKey;
    uint32_t enf, dz, tnf, tz;
    sel_block_scan2(nf, 0, enf, dz, tnf, tz, S);
    uint32_t pnf, pz, gnf, gz;
    sel_cluster_prefix2(cl, S, tnf, 0, pnf, pz, gnf, gz);
    A = static_cast<int32_t>(M < gnf ? M : gnf);
    uint32_t r = pnf + enf;
    for (int i = t0; i < t1 && r < static_cast<uint32_t>(A); ++i) {
      if (keys[i] != kFreeKey) continue;
      const int s = lo + i;
      const int32_t f = P.ws.miss_f[r];
      const int32_t h = P.ws.miss_h[r];
      keys[i] = kProtKey;
      P.pool.free_[s] = 0;
      P.pool.prio[s] = clock;
      P.pool.to_host[s] = h;
      P.pool.h2g[h] = s;
      P.pool.idxbuf[r] = s;
      P.ws.alloc_slot[r] = s;
      if (P.mode == kModeAlloc) P.out_slots[f] = s;
      ++r;
    }
    // misses beyond the free slots stay out of the pool
    const int gt = rank * kSelThreads + threadIdx.x;
    for (int rr = A + gt; rr < static_cast<int>(M); rr += C * kSelThreads) {
      const int32_t f = P.ws.miss_f[rr];
      P.pool.h2g[P.ws.miss_h[rr]] = kInf;
      if (P.mode == kModeRecall) P.ws.miss_stage[f] = -1;
      if (P.mode == kModeAlloc) P.out_slots[f] = -1;
    }
    if (static_cast<int32_t>(M) > A && rank == 0 && threadIdx.x == 0) set_status(P.status, ECHO_DEV_POOL_EXHAUSTED);
  }
  ECHO_TRACE_MARK(9);
  // -1 over the rest of the previous index list
  const int32_t list_len = P.mode == kModeEvict ? E : A;
  {
    const int gt = rank * kSelThreads + threadIdx.x;
    for (int i = list_len + gt; i < prev_idx && i < n_g; i += C * kSelThreads) P.pool.idxbuf[i] = -1;
  }
  cl.sync();
  if (rank == 0 && threadIdx.x == 0) {
    P.pool.counters[0] = n_free0 + E - A;
    P.pool.counters[1] = list_len;
    P.ws.ctr[kCtrMisses] = static_cast<int32_t>(M);
    P.ws.ctr[kCtrGranted] = A;
    if (P.stats) {
      auto add = [](int64_t *dst, unsigned long long v) {
        atomicAdd(reinterpret_cast<unsigned long long *>(dst), v);
      };
      if (P.mode == kModeRecall) {
        add(&P.stats->steps, 1ull);
        add(&P.stats->selected, n_sel);
        add(&P.stats->unique_rows, M + n_hit);
        add(&P.stats->hits, n_hit);
        add(&P.stats->misses, M);
        add(&P.stats->recalled, static_cast<unsigned long long>(A));
        add(&P.stats->unrecalled, static_cast<unsigned long long>(M - A));
      }
      if (P.mode == kModeAppend) add(&P.stats->appended, M);
      add(&P.stats->evicted, static_cast<unsigned long long>(E));
    }
  }
  if (P.stats && P.mode == kModeRecall && staged_total)
    atomicAdd(reinterpret_cast<unsigned long long *>(&P.stats->staged), static_cast<unsigned long long>(staged_total));
  ECHO_TRACE_MARK(10);
}

// ---------------------------------------------------------------------------
// copy: recalled / appended rows into their slots; out_slot of every entry
// ---------------------------------------------------------------------------
struct CopyParams {
  PoolView pool;
  Workspace ws;
  int mode;
  const uint16_t *stage_rows;  // recall: staged rows
  const uint16_t *new_kv;      // append: source rows by request
  // out_slot (recall)
  const int32_t *sel;
  const int32_t *req_to_host;
  int F, n_q, k, L_max;
  int32_t *out_slot;
  int32_t *stage_count;
  int B;
  echo_stats *stats;
};

constexpr int kCopyRows = 4;  // rows a warp moves at once (9 vectors in flight per lane)

__global__ void __launch_bounds__(256) copy_kernel(const CopyParams P) {
  const int lane = threadIdx.x & 31;
  const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nwarps = (gridDim.x * blockDim.x) >> 5;
  const int A = P.ws.ctr[kCtrGranted];
  const int4 *host = reinterpret_cast<const int4 *>(P.pool.host_kv);
  const int4 *stg = reinterpret_cast<const int4 *>(P.stage_rows);
  const int4 *newkv = reinterpret_cast<const int4 *>(P.new_kv);
  int4 *dst = reinterpret_cast<int4 *>(P.pool.gpu_kv);
  unsigned long long used = 0;
  for (int r0 = gwarp * kCopyRows; r0 < A; r0 += nwarps * kCopyRows) {
    const int n = A - r0 < kCopyRows ? A - r0 : kCopyRows;
    const int4 *src[kCopyRows];
    int32_t slot[kCopyRows];
#pragma unroll
    for (int r = 0; r < kCopyRows; ++r) {
      src[r] = nullptr;
      slot[r] = 0;
      if (r < n) {
        const int32_t f = P.ws.miss_f[r0 + r];
        slot[r] = P.ws.alloc_slot[r0 + r];
        if (P.mode == kModeAppend) {
          src[r] = newkv + static_cast<size_t>(f) * kKvChunks;
        } else {
          const int32_t st = P.ws.miss_stage[f];
          if (st >= 0) {
            src[r] = stg + static_cast<size_t>(st) * kKvChunks;
            used += lane == 0;
          } else {
            src[r] = host + static_cast<size_t>(P.ws.miss_h[r0 + r]) * kKvChunks;
          }
        }
      }
    }
    constexpr int kPer = (kCopyRows * kKvChunks + 31) / 32;
    int4 buf[kPer];
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int idx = m * 32 + lane;
      const int r = idx / kKvChunks, c = idx % kKvChunks;
      if (r < n) buf[m] = __ldcs(src[r] + c);
    }
#pragma unroll
    for (int m = 0; m < kPer; ++m) {
      const int idx = m * 32 + lane;
      const int r = idx / kKvChunks, c = idx % kKvChunks;
      if (r < n) dst[static_cast<size_t>(slot[r]) * kKvChunks + c] = buf[m];
    }
    if (P.mode == kModeRecall && lane < n) P.ws.miss_stage[P.ws.miss_f[r0 + lane]] = -1;
  }
  if (P.stats && used) atomicAdd(reinterpret_cast<unsigned long long *>(&P.stats->staged_used), used);

  if (P.mode == kModeRecall) {
    for (int f = blockIdx.x * blockDim.x + threadIdx.x; f < P.F; f += gridDim.x * blockDim.x) {
      const int32_t p = P.sel[f];
      int32_t o = -1;
      if (p >= 0 && p < P.L_max) {
        const int32_t h = P.req_to_host[static_cast<size_t>(f / (P.n_q * P.k)) * P.L_max + p];
        if (h >= 0 && h < P.pool.n_h) {
          const int32_t v = P.pool.h2g[h];
          o = (v >= 0 && v < P.pool.n_g) ? v : -1;
        }
      }
      P.out_slot[f] = o;
    }
    if (P.stage_count && blockIdx.x == 0)
      for (int b = threadIdx.x; b < P.B; b += blockDim.x) P.stage_count[b] = 0;
  }
}

// ---------------------------------------------------------------------------
// append: write-through of the generated token, then claim its host row
// ---------------------------------------------------------------------------
__global__ void append_prepare_kernel(PoolView pool, Workspace ws, uint8_t *k_index, int32_t *ctx_len,
                                      const int32_t *req_to_host, int B, int L_max, const uint16_t *new_kv,
                                      const uint8_t *new_k_index, int32_t *status) {
  const int b = blockIdx.x;
  if (b >= B) return;
  __shared__ int32_t sh_h, sh_p;
  if (threadIdx.x == 0) {
    const int32_t p = ctx_len[b];
    int32_t h = -1;
    if (p < 0 || p >= L_max) {
      set_status(status, ECHO_DEV_BAD_INDEX);
    } else {
      h = req_to_host[static_cast<size_t>(b) * L_max + p];
      if (h < 0 || h >= pool.n_h) {
        set_status(status, ECHO_DEV_BAD_INDEX);
        h = -1;
      }
    }
    sh_h = h;
    sh_p = p;
  }
  __syncthreads();
  const int32_t h = sh_h, p = sh_p;
  if (h >= 0) {
    // the host copy is written at generation (write-through), the GPU copy later by copy_kernel
    const int4 *src = reinterpret_cast<const int4 *>(new_kv) + static_cast<size_t>(b) * kKvChunks;
    int4 *hdst = reinterpret_cast<int4 *>(const_cast<uint16_t *>(pool.host_kv)) + static_cast<size_t>(h) * kKvChunks;
    for (int c = threadIdx.x; c < kKvChunks; c += blockDim.x) hdst[c] = src[c];
    const int4 *ksrc = reinterpret_cast<const int4 *>(new_k_index) + static_cast<size_t>(b) * (kDim / 16);
    int4 *kdst = reinterpret_cast<int4 *>(k_index + (static_cast<size_t>(b) * L_max + p) * kDim);
    for (int c = threadIdx.x; c < kDim / 16; c += blockDim.x) kdst[c] = ksrc[c];
  }
  if (threadIdx.x == 0) {
    ws.entry_rows[b] = h;
    if (h >= 0) {
      ctx_len[b] = p + 1;
      const int32_t v = pool.h2g[h];
      if (v != kInf && v >= 0) {
        set_status(status, ECHO_DEV_BAD_INDEX);  // the new token's row is already resident
        ws.entry_rows[b] = -1;
      } else {
        atomicMin(pool.h2g + h, kClaim + b);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// initialisation, EMA, clock
// ---------------------------------------------------------------------------
__global__ void pool_init_kernel(PoolView pool) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
  for (int s = tid; s < pool.n_g; s += nt) {
    pool.free_[s] = 1;
    pool.prio[s] = -1;
    pool.idxbuf[s] = -1;
    pool.to_host[s] = kInf;
  }
  for (int h = tid; h < pool.n_h; h += nt) pool.h2g[h] = kInf;
  if (tid == 0) {
    pool.counters[0] = pool.n_g;
    pool.counters[1] = 0;
    pool.counters[2] = 0;
    pool.counters[3] = 0;
  }
}

__global__ void ws_init_kernel(Workspace ws, int n_g, int max_rows) {
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
  for (int s = tid; s < n_g; s += nt) ws.slot_claim[s] = INT32_MAX;
  for (int i = tid; i < max_rows; i += nt) ws.miss_stage[i] = -1;
  for (int i = tid; i < kCtrCount; i += nt) ws.ctr[i] = 0;
}

__global__ void ema_kernel(float *s_hat, const float *kth, int n, float alpha, int32_t *clock_dev, int advance) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const float x = kth[i];
    if (isfinite(x)) {
      const float s = s_hat[i];
      if (isinf(s) && s > 0.f) {
        s_hat[i] = x;
      } else {
        const float a = __fmul_rn(alpha, s);
        const float c = __fmul_rn(__fsub_rn(1.0f, alpha), x);
        s_hat[i] = __fadd_rn(a, c);
      }
    }
  }
  if (i == 0 && clock_dev && advance) *clock_dev += 1;
}

}  // namespace echo

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
namespace echo_host {

int sm_count();

static echo::PoolView view_of(const echo_pool *p) {
  echo::PoolView v;
  v.free_ = p->gpu_token_free;
  v.prio = p->gpu_token_priority;
  v.idxbuf = p->gpu_indices_buffer;
  v.to_host = p->gpu_token_to_host;
  v.h2g = p->host_token_to_gpu;
  v.counters = p->counters;
  v.gpu_kv = p->gpu_kv;
  v.host_kv = p->host_kv;
  v.n_g = p->n_g;
  v.n_h = p->n_h;
  return v;
}

size_t workspace_bytes(int32_t n_g, int32_t max_rows) { return echo::ws_layout(n_g, max_rows, 0, nullptr); }

static echo::Workspace ws_of(const echo_workspace *w) {
  echo::Workspace x;
  echo::ws_layout(w->n_g, w->max_rows, reinterpret_cast<uintptr_t>(w->base), &x);
  return x;
}

static int grid_for(long long n, int block) {
  long long g = (n + block - 1) / block;
  long long cap = static_cast<long long>(sm_count()) * 8;
  if (g > cap) g = cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

static int check(const char *what) {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, what);
}

int launch_workspace_init(const echo_workspace *w, cudaStream_t s) {
  echo::ws_init_kernel<<<grid_for(w->n_g > w->max_rows ? w->n_g : w->max_rows, 256), 256, 0, s>>>(ws_of(w), w->n_g,
                                                                                                w->max_rows);
  return check("workspace init");
}

int launch_pool_init(const echo_pool *p, cudaStream_t s) {
  echo::pool_init_kernel<<<grid_for(p->n_h > p->n_g ? p->n_h : p->n_g, 256), 256, 0, s>>>(view_of(p));
  return check("pool init");
}

static echo::PlanParams base_params(const echo_pool *pool, const echo_workspace *ws, int mode, int32_t clock,
                                    const int32_t *clock_dev, int32_t *status) {
  echo::PlanParams P{};
  P.pool = view_of(pool);
  P.ws = ws_of(ws);
  P.mode = mode;
  P.clock = clock;
  P.clock_dev = clock_dev;
  P.status = status;
  P.cap_div = 1;
  P.stage_stride = 1;
  return P;
}

// one cluster of 8 CTAs (16 for pools above 8 x kPlanMaxChunk slots)
static int run_plan(const echo::PlanParams &P, cudaStream_t s) {
  const int C = P.pool.n_g <= 8 * echo::kPlanMaxChunk ? 8 : 16;
  const int chunk = (P.pool.n_g + C - 1) / C;
  if (chunk > echo::kPlanMaxChunk) {
    set_error("pool of %d slots exceeds the supported %d", P.pool.n_g, 16 * echo::kPlanMaxChunk);
    return ECHO_ENOTSUP;
  }
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(echo::plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(echo::plan_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e, "plan kernel attributes");
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C);
  cfg.blockDim = dim3(echo::kSelThreads);
  cfg.dynamicSmemBytes = sizeof(echo::SelSmem) + static_cast<size_t>(chunk) * sizeof(uint32_t);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, echo::plan_kernel, P);
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "cache-manager plan");
}

int launch_pool_alloc(const echo_pool *pool, const echo_workspace *ws, const int32_t *host_idx, const int32_t *n_dev,
                      int32_t max_n, int32_t clock, const int32_t *clock_dev, int32_t *out_slots, int32_t *status,
                      cudaStream_t s) {
  echo::PlanParams P = base_params(pool, ws, echo::kModeAlloc, clock, clock_dev, status);
  P.F = max_n;
  P.rows = host_idx;
  P.n_dev = n_dev;
  P.out_slots = out_slots;
  if (max_n > 0) {
    echo::claim_kernel<<<grid_for(max_n, 256), 256, 0, s>>>(P);
    int r = check("allocate claim");
    if (r) return r;
  }
  return run_plan(P, s);
}

int launch_pool_evict(const echo_pool *pool, const echo_workspace *ws, const int32_t *n_needed_dev, int32_t clock,
                      const int32_t *clock_dev, int32_t *status, cudaStream_t s) {
  echo::PlanParams P = base_params(pool, ws, echo::kModeEvict, clock, clock_dev, status);
  P.evict_n_dev = n_needed_dev;
  return run_plan(P, s);
}

int launch_recall(const echo_pool *pool, const echo_workspace *ws, const int32_t *sel, const int32_t *req_to_host,
                  const int32_t *ctx_len, int B, int n_q, int k, int L_max, const echo_stage *stage, int32_t clock,
                  const int32_t *clock_dev, int32_t *out_slot, echo_stats *stats, int32_t *status, cudaStream_t s) {
  echo::PlanParams P = base_params(pool, ws, echo::kModeRecall, clock, clock_dev, status);
  const int F = B * n_q * k;
  P.F = F;
  P.sel = sel;
  P.req_to_host = req_to_host;
  P.n_q = n_q;
  P.k = k;
  P.L_max = L_max;
  P.B = B;
  P.ctx_len = ctx_len;
  P.stats = stats;
  if (stage) {
    P.stage_host = stage->host_row;
    P.stage_count = stage->count;
    P.stage_stride = stage->stride;
    P.cap_div = stage->cap_div;
  }
  if (F > 0) {
    echo::claim_kernel<<<grid_for(F, 256), 256, 0, s>>>(P);
    int r = check("recall claim");
    if (r) return r;
  }
  int r = run_plan(P, s);
  if (r) return r;
  echo::CopyParams C{};
  C.pool = P.pool;
  C.ws = P.ws;
  C.mode = echo::kModeRecall;
  C.stage_rows = stage ? stage->rows : nullptr;
  C.sel = sel;
  C.req_to_host = req_to_host;
  C.F = F;
  C.n_q = n_q;
  C.k = k;
  C.L_max = L_max;
  C.out_slot = out_slot;
  C.stage_count = stage ? stage->count : nullptr;
  C.B = B;
  C.stats = stats;
  echo::copy_kernel<<<grid_for(F > 1024 ? F : 1024, 256), 256, 0, s>>>(C);
  return check("recall copy");
}

int launch_append(const echo_pool *pool, const echo_workspace *ws, uint8_t *k_index, int32_t *ctx_len,
                  const int32_t *req_to_host, int B, int L_max, const uint16_t *new_kv, const uint8_t *new_k_index,
                  int32_t clock, const int32_t *clock_dev, echo_stats *stats, int32_t *status, cudaStream_t s) {
  if (B == 0) return ECHO_OK;
  echo::PlanParams P = base_params(pool, ws, echo::kModeAppend, clock, clock_dev, status);
  P.F = B;
  P.rows = P.ws.entry_rows;
  P.stats = stats;
  echo::append_prepare_kernel<<<B, 128, 0, s>>>(P.pool, P.ws, k_index, ctx_len, req_to_host, B, L_max, new_kv,
                                                 new_k_index, status);
  int r = check("append prepare");
  if (r) return r;
  r = run_plan(P, s);
  if (r) return r;
  echo::CopyParams C{};
  C.pool = P.pool;
  C.ws = P.ws;
  C.mode = echo::kModeAppend;
  C.new_kv = new_kv;
  C.B = B;
  echo::copy_kernel<<<grid_for(B * 32, 256), 256, 0, s>>>(C);
  return check("append copy");
}

int launch_ema(float *s_hat, const float *kth, int n, float alpha, int32_t *clock_dev, int advance, cudaStream_t s) {
  echo::ema_kernel<<<(n + 255) / 256 > 0 ? (n + 255) / 256 : 1, 256, 0, s>>>(s_hat, kth, n, alpha, clock_dev, advance);
  return check("ema");
}

}  // namespace echo_host
