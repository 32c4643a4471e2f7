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
// sm_103a design: every operation (recall, allocate, evict, the append's
// allocation) is ONE cooperative kernel over all SMs, its phases separated by
// bounded grid barriers:
//   P1  (only when no earlier kernel did it) claims of the entries, see
//       cache_common.cuh; the decode step's top-k kernel claims what it selects.
//   P2  three warp roles at once: the slot scan (states cached in shared memory,
//       histogram of the evictable slots by age = clock - 1 - priority, 4096 bins,
//       the last one open-ended); the entries (classified as owned miss, repeat or
//       hit, hits' out_slot written, owned misses counted per CTA); the lookup of
//       the rows the prefetch staged.
//   P3  misses M = sum of the owned counts, evictions E = max(0, M - free); every
//       CTA finds the same threshold T (the E-th oldest priority, refined while the
//       open bin holds it); owned misses listed in entry order with their sources;
//       per-CTA counts of slots older than / at T and free.
//   P4  evictions and allocations together: prefix sums over the per-CTA counts
//       rank every free slot and every victim (slot order); the r-th of them takes
//       miss r.  The CTA that owns a slot writes all of it: the evicted row's map,
//       the new row's maps, priority = clock, indices-buffer entry, out_slot and the
//       KV row (16-byte vectors, 4 rows per warp, from the staging area or the
//       pinned host pool, read before the ranking so the host reads overlap it).
//       Every victim is taken (E never exceeds M - free), so no two CTAs write one
//       slot.  This is the page's ticket order taken in slot order: deterministic.
//   P5  only when a row was selected by several entries: after one more barrier,
//       the repeats take the slot of the row's first entry.
// Direct-to-slot prefetch (recall with a reserve): the slots the last recall set
// aside count as free here unless this step's prefetch filled them (P2's third role
// counts the filled ones and gives the unselected ones the step clock); E also
// covers the next reserve, and P4 hands the ranks after the misses' to it.
#include <atomic>

#include "cache_common.cuh"

ECHO_TRACE_UNIT(cache_mgr)

namespace echo {

enum Mode { kModeRecall = 0, kModeAlloc = 1, kModeAppend = 2, kModeEvict = 3 };

constexpr int kCoopThreads = 512;
constexpr int kCoopWarps = kCoopThreads / 32;

struct OpParams {
  PoolView pool;
  Workspace ws;
  int mode;
  int F;  // entries (recall: B * n_q * k; allocate: max_n; append: B)
  // recall entries
  const int32_t *sel;
  const int32_t *req_to_host;
  int n_q, k, L_max;
  // allocate / append entries
  const int32_t *rows;
  const int32_t *n_dev;
  int32_t *out_slots;
  // evict
  const int32_t *evict_n_dev;
  // staging (recall)
  const int32_t *stage_host;
  int32_t *stage_count;
  const uint16_t *stage_rows;
  const int32_t *ctx_len;
  int B, stage_stride, cap_div;
  // append: source rows
  const uint16_t *new_kv;
  // recall output
  int32_t *out_slot;
  int32_t clock;
  const int32_t *clock_dev;
  echo_stats *stats;
  int32_t *status;
  int claimed;  // recall: the entries were already claimed (by the top-k kernel)
  // decode step only: EMA of the k-th score and the device clock's advance
  float *s_hat;
  const float *kth;
  int n_ema;
  float alpha;
  int32_t *clock_advance;
  // shared-memory caches (entries per CTA they hold; 0 = not cached)
  int slot_cache_cap, ent_cache_cap;
  // direct-to-slot prefetch (recall; reserve != nullptr): slots set aside, [tickets
  // drawn, reserve length], slots to set aside for the next step
  int32_t *reserve;
  int32_t *reserve_ctl;
  int reserve_cap;
};

__device__ __forceinline__ int32_t read_clock(const OpParams &P) { return P.clock_dev ? *P.clock_dev : P.clock; }

// host row of entry f, or -1 (with BAD_INDEX flagged for out-of-range indices)
__device__ __forceinline__ int32_t entry_row(const OpParams &P, int f, int n_entries, bool flag) {
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

__device__ __forceinline__ int entries_count(const OpParams &P) {
  if (P.mode == kModeEvict) return 0;
  if (P.mode == kModeAlloc) {
    const int n = *P.n_dev;
    return n < 0 ? 0 : (n > P.F ? P.F : n);
  }
  return P.F;
}

// EMA of the k-th score (fp32, each operation rounded; +inf start takes kth)
__device__ __forceinline__ void ema_apply(float *s_hat, float x, float alpha) {
  if (!isfinite(x)) return;
  const float s = *s_hat;
  if (isinf(s) && s > 0.f) {
    *s_hat = x;
  } else {
    *s_hat = __fadd_rn(__fmul_rn(alpha, s), __fmul_rn(__fsub_rn(1.0f, alpha), x));
  }
}

__device__ __forceinline__ void ema_one(float *s_hat, const float *kth, int i, float alpha) {
  ema_apply(s_hat + i, kth[i], alpha);
}

__device__ __forceinline__ bool evictable(uint8_t fr, int32_t pr, int32_t clock) {
  return !fr && pr >= 0 && pr < clock;
}

// ---------------------------------------------------------------------------
// block-level helpers (kCoopThreads threads)
// ---------------------------------------------------------------------------
struct CoopSmem {
  uint32_t hist[kHistBins];
  uint32_t ws[4][kCoopWarps];
  uint32_t red[8];
  uint32_t pre[kCVals], tot[kCVals];
};

// exclusive block scan of NV counters; block totals in tot
template <int NV>
__device__ __forceinline__ void coop_scan(const uint32_t (&v)[NV], uint32_t (&ex)[NV], uint32_t (&tot)[NV],
                                          CoopSmem *S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) inc[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += u;
    }
  if (lane == 31)
#pragma unroll
    for (int k = 0; k < NV; ++k) S->ws[k][warp] = inc[k];
  __syncthreads();
  if (warp == 0)
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      uint32_t x = lane < kCoopWarps ? S->ws[k][lane] : 0u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      if (lane < kCoopWarps) S->ws[k][lane] = x;
    }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    ex[k] = (warp ? S->ws[k][warp - 1] : 0) + inc[k] - v[k];
    tot[k] = S->ws[k][kCoopWarps - 1];
  }
  __syncthreads();
}

// Bounded grid barrier of a cooperative launch (every CTA is resident), counted in
// two words of the workspace: an arrival count that is back at 0 between barriers
// and a generation number.  A CTA reads the generation, then arrives; the last of
// the G arrivals resets the count and publishes generation + 1, which the others
// wait for.  Nothing grows without bound (the generation compares by equality, so
// its wrap-around is harmless), so a workspace serves any number of calls.  A CTA
// that waits longer than kWaitLimitNs sets WAIT_TIMEOUT and reports failure; the
// caller then skips the remaining phases (the workspace must be re-initialised).
__device__ __forceinline__ bool grid_barrier(uint32_t *glob, int32_t *status, CoopSmem *S) {
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t ok = 1;
    const uint32_t G = gridDim.x;
    uint32_t gen, old;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(gen) : "l"(glob + kGGen) : "memory");
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(glob + kGBar) : "memory");
    if (old == G - 1) {
      // every CTA has arrived: the count restarts for the next barrier before this one opens
      asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(glob + kGBar), "r"(0u) : "memory");
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(glob + kGGen), "r"(gen + 1u) : "memory");
    } else {
      const uint64_t t0 = globaltimer();
      for (;;) {
        uint32_t cur;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(cur) : "l"(glob + kGGen) : "memory");
        if (cur != gen) break;
        if (globaltimer() - t0 > kWaitLimitNs) {
          set_status(status, ECHO_DEV_WAIT_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    S->red[7] = ok;
  }
  __syncthreads();
  return S->red[7] != 0;
}

// Adds a CTA's histogram into the global one.  Every CTA starts at a different
// 128-byte line, so the 152 CTAs' atomics spread over all lines at once instead of
// queueing on one line after another.
__device__ __forceinline__ void hist_flush(const uint32_t *local, uint32_t *global, int cta) {
  const int start = (cta * 32) & (kHistBins - 1);
  for (int k = threadIdx.x; k < kHistBins; k += kCoopThreads) {
    const int i = (k + start) & (kHistBins - 1);
    if (local[i]) red_add(global + i, local[i]);
  }
}

__device__ __forceinline__ void add_stat(echo_stats *st, int64_t echo_stats::*field, unsigned long long v) {
  if (st && v) red_add(reinterpret_cast<unsigned long long *>(&(st->*field)), v);
}

// ---------------------------------------------------------------------------
// the cooperative kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t slot_age(int32_t clock, int32_t pr) { return static_cast<uint32_t>(clock - 1 - pr); }

// The bin at which the running count of `gh` taken from the top bin down reaches
// `need`, and the count strictly above it (same answer in every CTA).
__device__ __forceinline__ void find_from_top(const uint32_t *gh, uint32_t need, uint32_t &bin, uint32_t &above,
                                              uint32_t &total, CoopSmem *S) {
  constexpr int per = kHistBins / kCoopThreads;  // 8 bins per thread, highest first
  uint32_t cnt[per];
  uint32_t mine = 0;
#pragma unroll
  for (int u = 0; u < per; ++u) {
    cnt[u] = __ldcg(gh + (kHistBins - 1 - (threadIdx.x * per + u)));
    mine += cnt[u];
  }
  uint32_t v1[1] = {mine}, ex1[1], tot1[1];
  coop_scan<1>(v1, ex1, tot1, S);
  total = tot1[0];
  uint32_t run = ex1[0];
#pragma unroll
  for (int u = 0; u < per; ++u) {
    if (run < need && run + cnt[u] >= need) {
      S->red[0] = static_cast<uint32_t>(kHistBins - 1 - (threadIdx.x * per + u));
      S->red[1] = run;
    }
    run += cnt[u];
  }
  __syncthreads();
  bin = S->red[0];
  above = S->red[1];
  __syncthreads();
}

constexpr int32_t kFreeMark = INT32_MIN;      // slot-cache value of a free slot
constexpr int32_t kResMark = INT32_MIN + 1;   // of a reserved slot the recall may hand out
constexpr int kSlotWarps = 8;              // P2 roles: slot scan, entries, staged rows
constexpr int kEntWarps = 6;
constexpr int kStageWarps = kCoopWarps - kSlotWarps - kEntWarps;
constexpr int kRows = 4;                   // KV rows a warp copies at once
constexpr uint32_t kSpreadMin = 2u * kCoopWarps * kRows;  // misses over which a CTA's copies may be spread
constexpr int kRowVecs = (kRows * kKvChunks + 31) / 32;  // 16-byte vectors per lane

// Loads of up to kRows KV rows (one warp): row u of the group comes from src[u].
__device__ __forceinline__ void rows_load(const int4 *const (&src)[kRows], int nr, int4 (&buf)[kRowVecs]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < kRowVecs; ++m) {
    const int idx = m * 32 + lane;
    const int u = idx / kKvChunks, ch = idx % kKvChunks;
    if (u < nr) buf[m] = __ldcs(pick_reg(src, u) + ch);
  }
}

__device__ __forceinline__ void rows_store(int4 *dst, const int32_t (&slot)[kRows], int n_keep,
                                           const int4 (&buf)[kRowVecs]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < kRowVecs; ++m) {
    const int idx = m * 32 + lane;
    const int u = idx / kKvChunks, ch = idx % kKvChunks;
    if (u < n_keep) dst[static_cast<size_t>(pick_reg(slot, u)) * kKvChunks + ch] = buf[m];
  }
}

// Source of the KV row of miss (entry f, host row h, staging index st): the
// generated token (append), the staging area, or the pinned host pool.
__device__ __forceinline__ const int4 *row_source(const OpParams &P, int32_t f, int32_t h, int32_t st) {
  const size_t rc = static_cast<size_t>(P.pool.row_chunks);
  if (P.mode == kModeAppend) return reinterpret_cast<const int4 *>(P.new_kv) + static_cast<size_t>(f) * rc;
  if (st >= 0) return reinterpret_cast<const int4 *>(P.stage_rows) + static_cast<size_t>(st) * kKvChunks;
  return reinterpret_cast<const int4 *>(P.pool.host_kv) + static_cast<size_t>(h) * rc;
}

// The rows of ranks [rbase, rbase + ntk) of the list of slots to take: slot maps,
// priority, indices-buffer entry and out_slot of each, and its KV bytes; warp w takes
// groups of kRows ranks from w * kRows on.  The slots come from tcache[t] (this CTA's
// own, cached at ranking) or the global alloc_slot.  use_first: each warp's first group
// was read before the ranking (entries, host rows, sources in my_*, latent bytes in
// buf).  Returns this lane's count of rows copied from the staging area.
__device__ __forceinline__ unsigned long long take_rows(const OpParams &P, int rbase, int ntk, const int32_t *tcache,
                                                        bool use_first, int my_t0, int32_t my_f, int32_t my_h,
                                                        int32_t my_src, int4 (&buf)[kRowVecs], int32_t clock,
                                                        bool copies, bool latent_rows) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long used = 0;
  for (int t0 = my_t0; t0 < ntk; t0 += kCoopWarps * kRows) {
    const int nr = min(kRows, ntk - t0);
    const bool first = use_first && t0 == my_t0;
    int32_t f = -1, h = -1, st = -1, s = -1;
    if (lane < nr) {
      const int r = rbase + t0 + lane;
      if (first) {
        f = my_f;
        h = my_h;
        st = my_src;
      } else {
        f = P.ws.miss_f[r];
        h = P.ws.miss_h[r];
        st = P.ws.miss_src[r];
      }
      s = tcache ? tcache[t0 + lane] : __ldcg(P.ws.alloc_slot + r);
      P.pool.free_[s] = 0;
      P.pool.prio[s] = clock;
      P.pool.to_host[s] = h;
      P.pool.h2g[h] = s;
      P.pool.idxbuf[r] = s;
      if (P.mode == kModeAlloc) P.out_slots[f] = s;
      if (P.mode == kModeRecall) {
        P.out_slot[f] = s;
        P.ws.miss_stage[f] = -1;  // staging lookup back to its resting state
        used += st >= 0;
      }
    }
    if (copies && latent_rows) {
      int32_t slot[kRows];
      const int4 *src[kRows];
#pragma unroll
      for (int u = 0; u < kRows; ++u) {
        slot[u] = __shfl_sync(0xffffffffu, s, u);
        const int32_t fu = __shfl_sync(0xffffffffu, f, u), hu = __shfl_sync(0xffffffffu, h, u),
                      su = __shfl_sync(0xffffffffu, st, u);
        src[u] = u < nr ? row_source(P, fu, hu, su) : nullptr;
      }
      if (!first) rows_load(src, nr, buf);
      rows_store(reinterpret_cast<int4 *>(P.pool.gpu_kv), slot, nr, buf);
    }
  }
  // rows of other lengths (block rows): every warp of the CTA copies 4 KB segments of
  // the rows it takes, so that a few large rows still keep all the warps'
  // loads in flight
  if (copies && !latent_rows && ntk > 0) {
    const int rc = P.pool.row_chunks;
    const int nseg = (rc + 32 * 8 - 1) / (32 * 8);
    int4 *kv = reinterpret_cast<int4 *>(P.pool.gpu_kv);
    for (int it = warp; it < ntk * nseg; it += kCoopWarps) {
      const int t = it / nseg, c0 = (it % nseg) * (32 * 8);
      const int r = rbase + t;
      const int32_t s = tcache ? tcache[t] : __ldcg(P.ws.alloc_slot + r);
      const int4 *src = row_source(P, P.ws.miss_f[r], P.ws.miss_h[r], P.ws.miss_src[r]);
      int4 *dst = kv + static_cast<size_t>(s) * rc;
      int4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = c0 + j * 32 + lane;
        if (i < rc) v[j] = __ldcs(src + i);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int i = c0 + j * 32 + lane;
        if (i < rc) dst[i] = v[j];
      }
    }
  }
  return used;
}

// The copies when some CTA may take many misses (a pool with free slots: the lowest
// free slots take the misses and sit in a few CTAs' ranges).  Every CTA computes every
// CTA's share from the per-CTA counts (thread r holds CTA r's: r_lt, r_eq, r_fr; the same
// numbers in every CTA); when the largest is over kSpreadMin and four times the mean,
// every CTA copies an even stripe of all ranks once every CTA has ranked its slots (one
// more grid barrier), else the owners copy their own.  Out of line, and the kernel's
// parameters in the constant bank (__grid_constant__, so that the reference to them
// needs no local copy): the full-pool path keeps the code it had.  Returns the lane's
// count of rows copied from the staging area, or ~0 when the grid barrier gave up.
__device__ __noinline__ unsigned long long spread_takes(const OpParams &P, CoopSmem *S, uint32_t *glob, uint32_t r_lt,
                                                       uint32_t r_eq, uint32_t r_fr, uint32_t needT, int32_t A,
                                                       uint32_t a_lo, int n_take, const int32_t *take_cache,
                                                       int32_t clock, bool copies, bool latent_rows) {
  const int G = gridDim.x, c = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t v3[3] = {r_lt, r_eq, r_fr}, ex3[3], tot3[3];
  coop_scan<3>(v3, ex3, tot3, S);
  uint32_t take = 0;
  if (static_cast<int>(threadIdx.x) < G) {
    const uint32_t alo = ex3[2] + ex3[0] + min(ex3[1], needT);
    const uint32_t nm = r_fr + r_lt + (min(ex3[1] + r_eq, needT) - min(ex3[1], needT));
    take = min(alo + nm, static_cast<uint32_t>(A)) - min(alo, static_cast<uint32_t>(A));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) take = max(take, __shfl_xor_sync(0xffffffffu, take, o));
  if (lane == 0) S->ws[0][warp] = take;
  __syncthreads();
  uint32_t mx = 0;
  for (int w = 0; w < kCoopWarps; ++w) mx = max(mx, S->ws[0][w]);
  __syncthreads();
  int rbase = static_cast<int>(a_lo), ntk = n_take;
  const int32_t *tcache = take_cache;
  if (mx > kSpreadMin && static_cast<unsigned long long>(mx) * G > 4ull * static_cast<uint32_t>(A)) {
    if (!grid_barrier(glob, P.status, S)) return ~0ull;
    const int per = (A + G - 1) / G;
    rbase = min(A, c * per);
    ntk = min(A, rbase + per) - rbase;
    tcache = nullptr;
  }
  int4 buf[kRowVecs];
  return take_rows(P, rbase, ntk, tcache, false, warp * kRows, -1, -1, -1, buf, clock, copies, latent_rows);
}

__global__ void __launch_bounds__(kCoopThreads, 1) cache_op_kernel(const __grid_constant__ OpParams P) {
  __shared__ CoopSmem S_;
  CoopSmem *S = &S_;
  extern __shared__ __align__(16) int32_t dyn_smem[];
  const int G = gridDim.x, c = blockIdx.x;
  const int gtid = c * kCoopThreads + threadIdx.x, gthreads = G * kCoopThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ECHO_TRACE_FIRST(24);
  pdl_wait();  // the selection and claims come from the kernel before (programmatic launch)
  ECHO_TRACE_FIRST(26);
  const int32_t clock = read_clock(P);
  const int n_g = P.pool.n_g;
  const int32_t n_free0 = P.pool.counters[0];
  const int32_t prev_idx = P.pool.counters[1];
  const int n = entries_count(P);
  uint32_t *glob = P.ws.glob;
  // direct to slot: the reserve and how many of its tickets the prefetch drew
  const bool direct = P.mode == kModeRecall && P.reserve != nullptr;
  int32_t res_len = 0, res_taken = 0;
  if (direct) {
    res_len = P.reserve_ctl[1];
    res_taken = min(P.reserve_ctl[0], res_len);
  }
  ECHO_TRACE_MARK(0);

  // this CTA's slots and entries (contiguous ranges, for the ordered phases)
  const int s_lo = static_cast<int>((static_cast<long long>(n_g) * c) / G);
  const int s_hi = static_cast<int>((static_cast<long long>(n_g) * (c + 1)) / G);
  const int e_lo = static_cast<int>((static_cast<long long>(n) * c) / G);
  const int e_hi = static_cast<int>((static_cast<long long>(n) * (c + 1)) / G);
  // shared-memory copies of the slot states (priority, kFreeMark if free) and of the
  // entries' classification, when they fit; the slots do not change from P2 to P4
  int32_t *slot_cache = (s_hi - s_lo) <= P.slot_cache_cap ? dyn_smem : nullptr;
  int32_t *host_cache = slot_cache ? dyn_smem + P.slot_cache_cap : nullptr;  // GPUTokenToHost of the slots
  int32_t *aux_cache = (e_hi - e_lo) <= P.ent_cache_cap ? dyn_smem + 2 * P.slot_cache_cap : nullptr;
  int32_t *h_cache = aux_cache ? aux_cache + P.ent_cache_cap : nullptr;     // host row of the entries
  // slots this CTA's phase P4 hands to misses, by rank (same capacity as the slot cache)
  int32_t *take_cache = slot_cache ? dyn_smem + 2 * P.slot_cache_cap + 2 * P.ent_cache_cap : nullptr;
  auto slot_val = [&](int s) -> int32_t {
    if (slot_cache) return slot_cache[s - s_lo];
    if (P.pool.free_[s]) return kFreeMark;
    const int32_t pr = P.pool.prio[s];
    return (direct && pr == kReservedPrio) ? kResMark : pr;
  };
  auto aux_of = [&](int f) -> int32_t { return aux_cache ? aux_cache[f - e_lo] : P.ws.ent_aux[f]; };
  const bool copies = P.mode == kModeRecall || P.mode == kModeAppend;

  // ===== P1: claims, unless the top-k kernel (recall) or the append already made them =====
  if ((P.mode == kModeRecall && !P.claimed) || P.mode == kModeAlloc) {
    for (int f = gtid; f < n; f += gthreads) {
      int32_t h = entry_row(P, f, n, true);
      if (P.mode == kModeAlloc) {
        if (h >= 0) {
          const int32_t v = P.pool.h2g[h];
          if (v != kInf && v >= 0) {  // already resident (or corrupt): cannot allocate again
            set_status(P.status, ECHO_DEV_BAD_INDEX);
            h = -1;
          } else {
            red_min(P.pool.h2g + h, kClaim + f);
          }
        }
        P.ws.entry_h[f] = h;
        if (h < 0) P.out_slots[f] = -1;
      } else {
        claim_entry(P.pool, P.ws, f, h, clock, P.status);
      }
    }
    ECHO_TRACE_MARK(1);
    if (!grid_barrier(glob, P.status, S)) return;
  }
  ECHO_TRACE_MARK(2);

  // ===== P2: three roles at once -- slot scan (states, age histogram), entries
  // (classification, out_slot of hits), staged-row lookup =====
  if (c == G - 1)  // the EMA needs only this step's k-th scores (complete before this kernel)
    for (int i = threadIdx.x; i < P.n_ema; i += kCoopThreads) ema_one(P.s_hat, P.kth, i, P.alpha);
  for (int i = threadIdx.x; i < kHistBins; i += kCoopThreads) S->hist[i] = 0;
  if (threadIdx.x < 8) S->red[threadIdx.x] = 0;
  __syncthreads();
  if (warp < kSlotWarps) {
    constexpr int kT = kSlotWarps * 32, kU = 8;  // one round of loads covers 2048 slots per CTA
    const bool hist_on = P.mode != kModeAlloc;
    for (int s0 = s_lo + static_cast<int>(threadIdx.x); s0 < s_hi; s0 += kT * kU) {
      uint8_t fr[kU];
      int32_t pr[kU], th[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int s = s0 + u * kT;
        fr[u] = 1;
        pr[u] = 0;
        th[u] = 0;
        if (s < s_hi) {
          fr[u] = P.pool.free_[s];
          pr[u] = P.pool.prio[s];
          if (host_cache) th[u] = P.pool.to_host[s];
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int s = s0 + u * kT;
        if (s >= s_hi) continue;
        const int32_t v = fr[u] ? kFreeMark : ((direct && pr[u] == kReservedPrio) ? kResMark : pr[u]);
        if (slot_cache) {
          slot_cache[s - s_lo] = v;
          host_cache[s - s_lo] = th[u];
        }
        if (hist_on && v >= 0 && v < clock) atomicAdd(&S->hist[min(slot_age(clock, v), kHistBins - 1u)], 1u);
      }
    }
    if (lane == 0) ECHO_TRACE_LAST_HERE(11);
  } else if (warp < kSlotWarps + kEntWarps) {
    if (P.mode != kModeEvict) {
      constexpr int kT = kEntWarps * 32, kU = 2;
      const int t = static_cast<int>(threadIdx.x) - kSlotWarps * 32;
      uint32_t own = 0, hits = 0, valid = 0, reps = 0;
      for (int f0 = e_lo + t; f0 < e_hi; f0 += kT * kU) {
        int32_t h[kU], v[kU], sc[kU];
        // recall: the claim recorded the map entry it saw, so a hit's slot (protected,
        // unchanged since) needs no second lookup; a miss reads the map for the winner
        const bool seen = P.mode == kModeRecall;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int f = f0 + u * kT;
          h[u] = -1;
          v[u] = kInf;
          if (f < e_hi) {
            h[u] = P.mode == kModeAppend ? P.ws.entry_rows[f] : P.ws.entry_h[f];
            if (seen) v[u] = P.ws.ent_aux[f];
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const bool hit = h[u] >= 0 && v[u] >= 0 && v[u] < n_g;
          sc[u] = -1;
          if (seen && hit) {
            sc[u] = P.ws.slot_claim[v[u]];
          } else if (h[u] >= 0) {
            v[u] = P.pool.h2g[h[u]];
          }
        }
        if (!seen) {
#pragma unroll
          for (int u = 0; u < kU; ++u)
            sc[u] = (h[u] >= 0 && v[u] >= 0 && v[u] < n_g) ? P.ws.slot_claim[v[u]] : -1;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int f = f0 + u * kT;
          if (f >= e_hi) continue;
          int32_t aux = -1;
          if (h[u] >= 0) {
            ++valid;
            if (v[u] == kClaim + f) {
              ++own;
              aux = -2;
            } else if (v[u] >= 0 && v[u] < n_g) {  // recall hit
              aux = v[u];
              if (sc[u] == f) {  // the first entry of the row: count it, clear its mark
                ++hits;
                P.ws.slot_claim[v[u]] = INT32_MAX;
              }
            } else if (v[u] < 0) {  // a repeat of a row an earlier entry claimed
              if (P.mode == kModeRecall) {
                aux = -3 - static_cast<int32_t>(static_cast<uint32_t>(v[u]) - 0x80000000u);
                ++reps;
              } else {
                if (P.mode == kModeAlloc) P.out_slots[f] = -1;
                set_status(P.status, ECHO_DEV_BAD_INDEX);
              }
            }
          }
          P.ws.ent_aux[f] = aux;
          if (aux_cache) {
            aux_cache[f - e_lo] = aux;
            h_cache[f - e_lo] = h[u];
          }
          if (P.mode == kModeRecall && aux >= -1) P.out_slot[f] = aux;  // hit slot, or -1
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        own += __shfl_xor_sync(0xffffffffu, own, o);
        hits += __shfl_xor_sync(0xffffffffu, hits, o);
        valid += __shfl_xor_sync(0xffffffffu, valid, o);
        reps += __shfl_xor_sync(0xffffffffu, reps, o);
      }
      if (lane == 0) {
        if (own) atomicAdd(&S->red[0], own);
        if (hits) atomicAdd(&S->red[1], hits);
        if (valid) atomicAdd(&S->red[2], valid);
        if (reps) atomicAdd(&S->red[3], reps);
      }
    }
    if (lane == 0) ECHO_TRACE_LAST_HERE(12);
  } else if (direct) {
    // the reserve slots this step's prefetch filled (a slot whose ticket lost the row
    // to another request's stays reserved); the unselected ones take the step clock
    const int t = static_cast<int>(threadIdx.x) - (kSlotWarps + kEntWarps) * 32;
    constexpr int kT = kStageWarps * 32;
    uint32_t filled = 0, used = 0;
    for (int i = c * kT + t; i < res_taken; i += G * kT) {
      const int32_t s = P.reserve[i];
      if (s < 0 || s >= n_g) continue;
      const int32_t pr = P.pool.prio[s];
      if (pr == kReservedPrio) continue;
      ++filled;
      if (pr == kPrefetchedPrio) {
        P.pool.prio[s] = clock;
      } else {
        ++used;  // selected: the claim gave it the clock
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      filled += __shfl_xor_sync(0xffffffffu, filled, o);
      used += __shfl_xor_sync(0xffffffffu, used, o);
    }
    if (lane == 0) {
      if (filled) atomicAdd(&S->red[4], filled);
      if (used) atomicAdd(&S->red[5], used);
    }
  } else if (P.mode == kModeRecall && P.stage_count != nullptr) {
    // which claimed misses the prefetch staged this step (one warp per request)
    const int sw = warp - kSlotWarps - kEntWarps;
    constexpr int kSpec = 4;  // staged rows per lane read together with the count
    for (int b = c * kStageWarps + sw; b < P.B; b += G * kStageWarps) {
      int L = P.ctx_len[b];
      int nb = P.stage_count[b];
      int32_t hs[kSpec];
#pragma unroll
      for (int j = 0; j < kSpec; ++j) {
        const int i = lane + 32 * j;
        hs[j] = i < P.stage_stride ? P.stage_host[static_cast<size_t>(b) * P.stage_stride + i] : -1;
      }
      L = L < 0 ? 0 : (L > P.L_max ? P.L_max : L);
      int cap = (L + P.cap_div - 1) / P.cap_div;
      cap = cap < P.stage_stride ? cap : P.stage_stride;
      nb = nb < cap ? nb : cap;
      // the first kSpec * 32 staged rows: all their map lookups in flight together
      int32_t vs[kSpec];
#pragma unroll
      for (int j = 0; j < kSpec; ++j) {
        const int i = lane + 32 * j;
        vs[j] = (i < nb && hs[j] >= 0 && hs[j] < P.pool.n_h) ? P.pool.h2g[hs[j]] : 0;
      }
#pragma unroll
      for (int j = 0; j < kSpec; ++j) {
        const int i = lane + 32 * j;
        if (i < nb && vs[j] < 0) {
          const uint32_t f = static_cast<uint32_t>(vs[j]) - 0x80000000u;  // v = kClaim + f
          if (f < static_cast<uint32_t>(P.F)) P.ws.miss_stage[f] = b * P.stage_stride + i;
        }
      }
      for (int i = lane + 32 * kSpec; i < nb; i += 32) {  // beyond: one at a time
        const int32_t h = P.stage_host[static_cast<size_t>(b) * P.stage_stride + i];
        if (h < 0 || h >= P.pool.n_h) continue;
        const int32_t v = P.pool.h2g[h];
        if (v < 0) {
          const uint32_t f = static_cast<uint32_t>(v) - 0x80000000u;
          if (f < static_cast<uint32_t>(P.F)) P.ws.miss_stage[f] = b * P.stage_stride + i;
        }
      }
      if (lane == 0) add_stat(P.stats, &echo_stats::staged, static_cast<unsigned long long>(nb));
    }
    if (lane == 0) ECHO_TRACE_LAST_HERE(13);
  }
  __syncthreads();
  if (P.mode != kModeAlloc) hist_flush(S->hist, P.ws.hist, c);
  if (threadIdx.x == 0 && P.mode != kModeEvict) {
    P.ws.cta[c * kCVals + kCOwn] = S->red[0];
    if (S->red[1]) red_add(glob + kGHits, S->red[1]);
    if (S->red[2]) red_add(glob + kGValid, S->red[2]);
    if (S->red[3]) red_add(glob + kGRepeats, S->red[3]);
    if (S->red[4]) red_add(glob + kGFilled, S->red[4]);
    add_stat(P.stats, &echo_stats::staged, S->red[4]);
    add_stat(P.stats, &echo_stats::staged_used, S->red[5]);
  }
  ECHO_TRACE_MARK(3);
  if (!grid_barrier(glob, P.status, S)) return;
  ECHO_TRACE_MARK(4);

  // ===== P3: M, E, threshold; owned misses listed in entry order; per-CTA slot counts =====
  // the global words, the per-CTA owned counts and the age histogram (highest bin
  // first) load together
  uint32_t g_valid = 0, g_hits = 0, g_rep = 0, g_fill = 0;
  if (threadIdx.x == 0) {
    if (c == 0) {
      g_valid = __ldcg(glob + kGValid);
      g_hits = __ldcg(glob + kGHits);
    }
    g_rep = P.mode == kModeRecall ? __ldcg(glob + kGRepeats) : 0u;
    g_fill = direct ? __ldcg(glob + kGFilled) : 0u;
  }
  constexpr int kPerBin = kHistBins / kCoopThreads;
  uint32_t hcnt[kPerBin];
  uint32_t m = 0, pm = 0, hmine = 0;
  if (P.mode != kModeEvict)
    for (int r = threadIdx.x; r < G; r += kCoopThreads) {
      const uint32_t x = __ldcg(P.ws.cta + r * kCVals + kCOwn);
      m += x;
      if (r < c) pm += x;
    }
#pragma unroll
  for (int u = 0; u < kPerBin; ++u) {
    hcnt[u] = P.mode != kModeAlloc ? __ldcg(P.ws.hist + (kHistBins - 1 - (threadIdx.x * kPerBin + u))) : 0u;
    hmine += hcnt[u];
  }
  // final after the barrier: the step's valid entries and hits (for the stats); repeats
  // of a missed row need one more grid barrier (thread 0 read the count, the scan below
  // hands it to the rest)
  if (threadIdx.x == 0) {
    if (c == 0) {
      glob[kGValid] = 0;
      glob[kGHits] = 0;
    }
    S->red[6] = g_rep;
    S->red[5] = g_fill;
  }
  // this thread's segment of the entries; the staging rows of its owned misses
  const int e_cnt = e_hi - e_lo;
  const int e_per = (e_cnt + kCoopThreads - 1) / kCoopThreads;
  const int ef0 = e_lo + min(e_cnt, static_cast<int>(threadIdx.x) * e_per);
  const int ef1 = e_lo + min(e_cnt, static_cast<int>(threadIdx.x + 1) * e_per);
  constexpr int kStg = 8;
  int32_t stg[kStg];
#pragma unroll
  for (int u = 0; u < kStg; ++u)
    stg[u] = (P.mode == kModeRecall && ef0 + u < ef1 && aux_of(ef0 + u) == -2) ? P.ws.miss_stage[ef0 + u] : -1;
  // this thread's owned misses (their ranks follow the same scan)
  uint32_t own_seg = 0;
  if (P.mode != kModeEvict)
    for (int f = ef0; f < ef1; ++f) own_seg += aux_of(f) == -2;
  uint32_t M = 0, pre_own = 0, hist_total = 0, hist_ex = 0, own_ex = 0;
  {
    uint32_t v4[4] = {m, pm, hmine, own_seg}, ex4[4], tot4[4];
    coop_scan<4>(v4, ex4, tot4, S);
    M = tot4[0];
    pre_own = tot4[1];
    hist_total = tot4[2];
    hist_ex = ex4[2];
    own_ex = ex4[3];
  }
  const bool any_repeats = S->red[6] != 0;  // written before the scan's barriers
  // direct to slot: reserved slots the prefetch left unused return to the free ones
  const int32_t released = direct ? res_len - static_cast<int32_t>(S->red[5]) : 0;
  const int32_t res_want = direct ? max(P.reserve_cap, 0) : 0;
  ECHO_TRACE_MARK(14);
  int32_t E = 0;
  if (P.mode == kModeEvict) {
    E = *P.evict_n_dev;
    E = E < 0 ? 0 : E;
  } else if (P.mode != kModeAlloc) {
    // direct to slot: evict for the next reserve too
    E = static_cast<int32_t>(M) + res_want - (n_free0 + released);
    E = E < 0 ? 0 : E;
  }
  if (E > 0 && hist_total < static_cast<uint32_t>(E)) {  // fewer evictable slots than asked
    // (a short reserve is no exhaustion: misses left out are flagged after P4)
    if (c == 0 && threadIdx.x == 0 && !direct) set_status(P.status, ECHO_DEV_POOL_EXHAUSTED);
    E = static_cast<int32_t>(hist_total);
  }
  int32_t Tp = 0;  // threshold priority: victims have priority < Tp, or == Tp (the first needT)
  uint32_t needT = 0;
  if (E > 0) {
    // the age bin where the count from the oldest bin down reaches E
    uint32_t run = hist_ex;
#pragma unroll
    for (int u = 0; u < kPerBin; ++u) {
      if (run < static_cast<uint32_t>(E) && run + hcnt[u] >= static_cast<uint32_t>(E)) {
        S->red[0] = static_cast<uint32_t>(kHistBins - 1 - (threadIdx.x * kPerBin + u));
        S->red[1] = run;
      }
      run += hcnt[u];
    }
    __syncthreads();
    const uint32_t d = S->red[0], above = S->red[1];
    __syncthreads();
    uint32_t need = static_cast<uint32_t>(E) - above;
    uint32_t age_t = d;
    if (d == kHistBins - 1) {
      // the open bin (age >= 4095): refine x = age - 4095 by 12-bit digits, oldest first
      const uint32_t xmax = static_cast<uint32_t>(clock) - static_cast<uint32_t>(kHistBins);
      int hb = xmax == 0 ? 0 : 32 - __clz(xmax);
      uint32_t prefix = 0;
      for (int lvl = 1; hb > 0; ++lvl) {
        const int width = hb < 12 ? hb : 12;
        const int sh = hb - width;
        for (int i = threadIdx.x; i < kHistBins; i += kCoopThreads) S->hist[i] = 0;
        __syncthreads();
        for (int s = s_lo + threadIdx.x; s < s_hi; s += kCoopThreads) {
          const int32_t pr = slot_val(s);
          if (!(pr >= 0 && pr < clock)) continue;
          const uint32_t age = slot_age(clock, pr);
          if (age < kHistBins - 1u) continue;
          const uint32_t x = age - (kHistBins - 1u);
          if (hb < 32 && (x >> hb) != (prefix >> hb)) continue;
          atomicAdd(&S->hist[(x >> sh) & ((1u << width) - 1u)], 1u);
        }
        __syncthreads();
        uint32_t *gl = P.ws.hist + lvl * kHistBins;
        hist_flush(S->hist, gl, c);
        if (!grid_barrier(glob, P.status, S)) return;
        uint32_t dd, ab, tt;
        find_from_top(gl, need, dd, ab, tt, S);
        prefix |= dd << sh;
        need -= ab;
        hb = sh;
      }
      age_t = (kHistBins - 1u) + prefix;
    }
    Tp = clock - 1 - static_cast<int32_t>(age_t);
    needT = need;
  }
  ECHO_TRACE_MARK(15);
  uint32_t my_lt = 0, my_eq = 0, my_fr = 0;  // this CTA's slots older than / at T, free
  // owned misses, in entry order (contiguous per-thread segments), with their sources
  if (P.mode != kModeEvict) {
    uint32_t r = pre_own + own_ex;
#pragma unroll
    for (int u = 0; u < kStg; ++u) {
      const int f = ef0 + u;
      if (f >= ef1 || aux_of(f) != -2) continue;
      P.ws.miss_f[r] = f;
      P.ws.miss_h[r] = h_cache ? h_cache[f - e_lo] : (P.mode == kModeAppend ? P.ws.entry_rows[f] : P.ws.entry_h[f]);
      P.ws.miss_src[r] = stg[u];
      P.ws.miss_rank[f] = static_cast<int32_t>(r);
      ++r;
    }
    for (int f = ef0 + kStg; f < ef1; ++f) {
      if (aux_of(f) != -2) continue;
      P.ws.miss_f[r] = f;
      P.ws.miss_h[r] = h_cache ? h_cache[f - e_lo] : (P.mode == kModeAppend ? P.ws.entry_rows[f] : P.ws.entry_h[f]);
      P.ws.miss_src[r] = P.mode == kModeRecall ? P.ws.miss_stage[f] : -1;
      P.ws.miss_rank[f] = static_cast<int32_t>(r);
      ++r;
    }
  }
  // this CTA's slots older than / at T and free, counted over contiguous per-thread
  // segments: the exclusive prefixes stay in registers for phase P4's ranking
  const int s_cnt = s_hi - s_lo;
  const int s_per = (s_cnt + kCoopThreads - 1) / kCoopThreads;
  const int q0 = s_lo + min(s_cnt, static_cast<int>(threadIdx.x) * s_per);
  const int q1 = s_lo + min(s_cnt, static_cast<int>(threadIdx.x + 1) * s_per);
  uint32_t seg_lt_ex = 0, seg_eq_ex = 0, seg_fr_ex = 0;
  {
    uint32_t lt = 0, eq = 0, fr = 0;
    for (int s = q0; s < q1; ++s) {
      const int32_t v = slot_val(s);
      if (v == kFreeMark || v == kResMark) {
        ++fr;
      } else if (E > 0 && v >= 0 && v < clock) {
        lt += v < Tp;
        eq += v == Tp;
      }
    }
    uint32_t v3[3] = {lt, eq, fr}, ex3[3], tot3[3];
    coop_scan<3>(v3, ex3, tot3, S);
    seg_lt_ex = ex3[0];
    seg_eq_ex = ex3[1];
    seg_fr_ex = ex3[2];
    my_lt = tot3[0];
    my_eq = tot3[1];
    my_fr = tot3[2];
    if (threadIdx.x == 0) {
      P.ws.cta[c * kCVals + kCLt] = tot3[0];
      P.ws.cta[c * kCVals + kCEq] = tot3[1];
      P.ws.cta[c * kCVals + kCFree] = tot3[2];
    }
  }
  ECHO_TRACE_MARK(5);
  if (!grid_barrier(glob, P.status, S)) return;
  ECHO_TRACE_MARK(6);

  // ===== P4: evictions and allocations together.  Free slots and victims, in slot
  // order, form the list of slots to take; the r-th of them takes miss r.  The CTA
  // that owns a slot ranks it and clears the evicted row's map; the CTA that copies
  // rank r (the slot's owner, or, when a few CTAs hold most of the slots to take, the
  // CTA whose even stripe of the ranks holds r) writes the rest: the new row's maps,
  // priority, indices-buffer entry, out_slot and KV bytes =====
  uint32_t pre_lt = 0, pre_eq = 0, pre_fr = 0, free_total = 0;
  uint32_t r_lt = 0, r_eq = 0, r_fr = 0;  // the counts of CTA r = threadIdx.x (when G <= the CTA's threads)
  uint32_t n_big = 0;  // CTAs whose candidate slots are more than kSpreadMin: only they can take that many
  {
    uint32_t a3[3] = {0, 0, 0}, t1 = 0, big = 0;
    for (int r = threadIdx.x; r < G; r += kCoopThreads) {
      const uint32_t lt = __ldcg(P.ws.cta + r * kCVals + kCLt), eq = __ldcg(P.ws.cta + r * kCVals + kCEq),
                     fr = __ldcg(P.ws.cta + r * kCVals + kCFree);
      if (r == static_cast<int>(threadIdx.x)) {
        r_lt = lt;
        r_eq = eq;
        r_fr = fr;
      }
      if (r < c) {
        a3[0] += lt;
        a3[1] += eq;
        a3[2] += fr;
      }
      t1 += fr;
      big += lt + eq + fr > kSpreadMin;
    }
    uint32_t v5[5] = {a3[0], a3[1], a3[2], t1, big}, ex5[5], tot5[5];
    coop_scan<5>(v5, ex5, tot5, S);
    pre_lt = tot5[0];
    pre_eq = tot5[1];
    pre_fr = tot5[2];
    free_total = tot5[3];
    n_big = tot5[4];
  }
  const int32_t A = (P.mode == kModeEvict) ? 0 : static_cast<int32_t>(min(M, free_total + static_cast<uint32_t>(E)));
  // the next reserve: the ranks after the misses'
  const int32_t R = min(res_want, static_cast<int32_t>(free_total + static_cast<uint32_t>(E)) - A);
  // this CTA's slots to take have ranks [a_lo, a_lo + n_mine); those below A get a miss
  const uint32_t a_lo = pre_fr + pre_lt + min(pre_eq, needT);
  const uint32_t n_mine = my_fr + my_lt + (min(pre_eq + my_eq, needT) - min(pre_eq, needT));
  const int n_take = static_cast<int>(min(a_lo + n_mine, static_cast<uint32_t>(A)) - min(a_lo, static_cast<uint32_t>(A)));
  // Where the copies fall: when some CTA may take more than kSpreadMin misses (a pool
  // with free slots, whose lowest free slots take the misses and sit in a few CTAs'
  // ranges; or victims bunched in a few ranges), the copies may be spread over the
  // grid after the ranking.  Otherwise (victims scattered over all CTAs) the slots'
  // owners copy, and the first rows are loaded before the ranking.
  const bool may_spread = copies && G <= kCoopThreads && A > static_cast<int32_t>(kSpreadMin) && n_big > 0;
  // each warp's first four misses: entry, host row, source, and the KV rows themselves,
  // loaded now so that the host reads overlap the ranking below (not when the copies
  // may be spread)
  int4 buf[kRowVecs];
  int32_t my_f = -1, my_h = -1, my_src = -1;  // lane u < kRows: rank a_lo + warp * kRows + u
  const int my_t0 = warp * kRows;
  const int my_nr = (!may_spread && n_take > my_t0) ? min(kRows, n_take - my_t0) : 0;
  if (lane < my_nr) {
    const int r = static_cast<int>(a_lo) + my_t0 + lane;
    my_f = P.ws.miss_f[r];
    my_h = P.ws.miss_h[r];
    my_src = P.ws.miss_src[r];
  }
  const bool latent_rows = P.pool.row_chunks == kKvChunks;  // rows of other lengths copy after the ranking
  if (copies && latent_rows && my_nr > 0) {
    const int4 *src[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int32_t f = __shfl_sync(0xffffffffu, my_f, u), h = __shfl_sync(0xffffffffu, my_h, u),
                    st = __shfl_sync(0xffffffffu, my_src, u);
      src[u] = u < my_nr ? row_source(P, f, h, st) : nullptr;
    }
    rows_load(src, my_nr, buf);
  }
  // rank this CTA's slots (the per-thread segments and prefixes of P3); victims lose
  // their maps
  {
    uint32_t lt_b = pre_lt + seg_lt_ex, eq_b = pre_eq + seg_eq_ex, fr_b = pre_fr + seg_fr_ex;
    for (int s = q0; s < q1; ++s) {
      const int32_t v = slot_val(s);
      // victims before s (all evictable slots older than T, the first needT at T), and
      // the slots to take before s (free ones and victims)
      const uint32_t vb = lt_b + min(eq_b, needT);
      const uint32_t before = fr_b + vb;
      if (v == kFreeMark || v == kResMark) {
        if (before < static_cast<uint32_t>(A)) {
          P.ws.alloc_slot[before] = s;
          if (take_cache) take_cache[before - a_lo] = s;
        } else if (before < static_cast<uint32_t>(A + R)) {  // into the next reserve
          P.reserve[before - A] = s;
          if (v == kFreeMark) {
            P.pool.free_[s] = 0;
            P.pool.prio[s] = kReservedPrio;
          }
        } else if (v == kResMark) {  // an unused reserved slot nobody takes: free
          P.pool.free_[s] = 1;
          P.pool.prio[s] = -1;
        }
        ++fr_b;
        continue;
      }
      if (E == 0 || !(v >= 0 && v < clock)) continue;
      bool victim = false;
      if (v < Tp) {
        victim = true;
        ++lt_b;
      } else if (v == Tp) {
        victim = eq_b < needT;
        ++eq_b;
      }
      if (!victim) continue;
      const int32_t h = host_cache ? host_cache[s - s_lo] : P.pool.to_host[s];
      if (h >= 0 && h < P.pool.n_h) P.pool.h2g[h] = kInf;
      if (P.mode == kModeEvict) P.pool.idxbuf[vb] = s;  // evicted slots in ascending order
      if (before < static_cast<uint32_t>(A)) {
        P.ws.alloc_slot[before] = s;
        if (take_cache) take_cache[before - a_lo] = s;
      } else if (before < static_cast<uint32_t>(A + R)) {  // into the next reserve
        P.reserve[before - A] = s;
        P.pool.prio[s] = kReservedPrio;
        P.pool.to_host[s] = kInf;
      } else {  // nobody takes it: free
        P.pool.free_[s] = 1;
        P.pool.prio[s] = -1;
        P.pool.to_host[s] = kInf;
      }
    }
  }
  __syncthreads();  // this CTA's slot table complete
  ECHO_TRACE_MARK(7);
  unsigned long long used = 0;
  if (!may_spread) {
    // the misses this CTA's slots take: four per warp (the first four already loaded)
    used = take_rows(P, static_cast<int>(a_lo), n_take, take_cache, true, my_t0, my_f, my_h, my_src, buf, clock,
                     copies, latent_rows);
  } else {
    // the owners' copies, or an even stripe per CTA (spread_takes decides)
    used = spread_takes(P, S, glob, r_lt, r_eq, r_fr, needT, A, a_lo, n_take, take_cache, clock, copies, latent_rows);
    if (used == ~0ull) return;
  }
  // misses beyond the pool's capacity stay out of it
  for (int r = A + gtid; r < static_cast<int>(M); r += gthreads) {
    const int32_t f = P.ws.miss_f[r], h = P.ws.miss_h[r];
    P.pool.h2g[h] = kInf;
    if (P.mode == kModeRecall) {
      P.out_slot[f] = -1;
      P.ws.miss_stage[f] = -1;
    }
    if (P.mode == kModeAlloc) P.out_slots[f] = -1;
  }
  ECHO_TRACE_MARK(8);
  if (any_repeats) {
    // repeats of a missed row take the slot of the row's first entry
    if (!grid_barrier(glob, P.status, S)) return;
    for (int f = e_lo + static_cast<int>(threadIdx.x); f < e_hi; f += kCoopThreads) {
      const int32_t aux = aux_of(f);
      if (aux > -3) continue;
      const int32_t r1 = P.ws.miss_rank[-3 - aux];
      P.out_slot[f] = r1 < A ? __ldcg(P.ws.alloc_slot + r1) : -1;
    }
    if (c == 0 && threadIdx.x == 0) glob[kGRepeats] = 0;  // every CTA read it before the barrier
  }
  if (static_cast<int32_t>(M) > A && c == 0 && threadIdx.x == 0) set_status(P.status, ECHO_DEV_POOL_EXHAUSTED);
  const int32_t list_len = P.mode == kModeEvict ? E : A;
  for (int i = list_len + gtid; i < prev_idx && i < n_g; i += gthreads) P.pool.idxbuf[i] = -1;
  if (P.mode == kModeRecall) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) used += __shfl_xor_sync(0xffffffffu, used, o);
    if (lane == 0) add_stat(P.stats, &echo_stats::staged_used, used);
  }
  // scratch back to its resting state (nothing reads it any more)
  for (int i = gtid; i < kHistLevels * kHistBins; i += gthreads) P.ws.hist[i] = 0;
  if (c == 0 && threadIdx.x == 0) {
    P.pool.counters[0] = n_free0 + released + E - A - R;
    P.pool.counters[1] = list_len;
    if (direct) {  // every CTA read these at its start and the filled count after P2
      P.reserve_ctl[0] = 0;
      P.reserve_ctl[1] = R;
      glob[kGFilled] = 0;
    }
    P.ws.ctr[kCtrMisses] = static_cast<int32_t>(M);
    P.ws.ctr[kCtrGranted] = A;
    const uint32_t valid = g_valid, hits = g_hits;
    if (P.mode == kModeRecall) {
      add_stat(P.stats, &echo_stats::steps, 1ull);
      add_stat(P.stats, &echo_stats::selected, valid);
      add_stat(P.stats, &echo_stats::unique_rows, static_cast<unsigned long long>(M) + hits);
      add_stat(P.stats, &echo_stats::hits, hits);
      add_stat(P.stats, &echo_stats::misses, M);
      add_stat(P.stats, &echo_stats::recalled, static_cast<unsigned long long>(A));
      add_stat(P.stats, &echo_stats::unrecalled, static_cast<unsigned long long>(M - A));
    }
    if (P.mode == kModeAppend) add_stat(P.stats, &echo_stats::appended, M);
    add_stat(P.stats, &echo_stats::evicted, static_cast<unsigned long long>(E));
    if (P.clock_advance) *P.clock_advance = clock + 1;  // every CTA read the clock at its start
  }
  if (c == 0 && P.mode == kModeRecall && P.stage_count)
    for (int b = threadIdx.x; b < P.B; b += kCoopThreads) P.stage_count[b] = 0;
  ECHO_TRACE_MARK(9);
  ECHO_TRACE_LAST(25);
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
    // the host copy is written at generation (write-through); the GPU copy follows
    // in the allocation kernel
    const int rc = pool.row_chunks;
    const int4 *src = reinterpret_cast<const int4 *>(new_kv) + static_cast<size_t>(b) * rc;
    int4 *hdst = reinterpret_cast<int4 *>(const_cast<uint16_t *>(pool.host_kv)) + static_cast<size_t>(h) * rc;
    for (int i = threadIdx.x; i < rc; i += blockDim.x) hdst[i] = src[i];
    const int4 *ksrc = reinterpret_cast<const int4 *>(new_k_index) + static_cast<size_t>(b) * (kDim / 16);
    int4 *kdst = reinterpret_cast<int4 *>(k_index + (static_cast<size_t>(b) * L_max + p) * kDim);
    for (int i = threadIdx.x; i < kDim / 16; i += blockDim.x) kdst[i] = ksrc[i];
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
        red_min(pool.h2g + h, kClaim + b);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// initialisation, EMA
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
  for (int i = tid; i < kHistLevels * kHistBins; i += nt) ws.hist[i] = 0;
  for (int i = tid; i < kMaxGrid * kCVals; i += nt) ws.cta[i] = 0;
  for (int i = tid; i < kGCount; i += nt) ws.glob[i] = 0u;
  for (int i = tid; i < kCtrCount; i += nt) ws.ctr[i] = 0;
  for (int i = tid; i < kSelHintRows * kSelBins; i += nt) ws.sel_hist[i] = 0;
  for (int i = tid; i < kSelHintRows; i += nt) ws.sel_hint[i] = make_int4(0, 0, 0, 0);
}

// Self-test of the bounded waits (no counterpart on the pages).  which = 0: one
// thread waits on an mbarrier nothing arrives on; which = 1: a cooperative grid
// barrier that CTA 0 never reaches.  Either wait gives up after kWaitLimitNs and sets
// WAIT_TIMEOUT; every CTA returns, so the context stays usable.
__global__ void __launch_bounds__(kCoopThreads, 1) wait_probe_kernel(int which, uint32_t *glob, int32_t *status) {
  __shared__ CoopSmem S_;
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (which == 0) {
    if (blockIdx.x != 0) return;
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1);
      abort_flag = 0;
      fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status);
    return;
  }
  if (blockIdx.x == 0) return;  // the CTA the others wait for
  grid_barrier(glob, status, &S_);
}

__global__ void ema_kernel(float *s_hat, const float *kth, int n, int stride, float alpha) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) ema_apply(s_hat + i, kth[static_cast<size_t>(i) * stride], alpha);
}

}  // namespace echo

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
namespace echo_host {

int sm_count();

echo::PoolView pool_view(const echo_pool *p);
echo::Workspace workspace_view(const echo_workspace *w);

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
  v.row_chunks = (p->row_elems > 0 ? p->row_elems : echo::kKvElems) / 8;
  return v;
}

size_t workspace_bytes(int32_t n_g, int32_t max_rows) { return echo::ws_layout(n_g, max_rows, 0, nullptr); }

echo::PoolView pool_view(const echo_pool *p) { return view_of(p); }

static echo::Workspace ws_of(const echo_workspace *w) {
  echo::Workspace x;
  echo::ws_layout(w->n_g, w->max_rows, reinterpret_cast<uintptr_t>(w->base), &x);
  return x;
}

echo::Workspace workspace_view(const echo_workspace *w) { return ws_of(w); }

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
  const int n = w->n_g > w->max_rows ? w->n_g : w->max_rows;
  echo::ws_init_kernel<<<grid_for(n > 65536 ? n : 65536, 256), 256, 0, s>>>(ws_of(w), w->n_g, w->max_rows);
  return check("workspace init");
}

int launch_pool_init(const echo_pool *p, cudaStream_t s) {
  echo::pool_init_kernel<<<grid_for(p->n_h > p->n_g ? p->n_h : p->n_g, 256), 256, 0, s>>>(view_of(p));
  return check("pool init");
}

static echo::OpParams base_params(const echo_pool *pool, const echo_workspace *ws, int mode, int32_t clock,
                                  const int32_t *clock_dev, int32_t *status) {
  echo::OpParams P{};
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

// one cooperative launch over all SMs (one CTA each); `pdl`: programmatic launch
// after the kernel before it on the stream
constexpr int kSlotCacheMax = 12288;  // slots per CTA whose states P2 keeps in shared memory
constexpr int kEntCacheMax = 4096;    // entries per CTA whose classification P2 keeps

static int run_op(const echo::OpParams &P0, cudaStream_t s, bool pdl = false) {
  const int grid = sm_count() < echo::kMaxGrid ? sm_count() : echo::kMaxGrid;
  echo::OpParams P = P0;
  const long long spc = (static_cast<long long>(P.pool.n_g) + grid - 1) / grid;
  const long long epc = (static_cast<long long>(P.mode == echo::kModeEvict ? 0 : P.F) + grid - 1) / grid;
  P.slot_cache_cap = spc <= kSlotCacheMax ? static_cast<int>(spc) : 0;
  P.ent_cache_cap = epc <= kEntCacheMax ? static_cast<int>(epc) : 0;
  static std::atomic<bool> attr[kMaxDevices];
  if (int r = smem_limit_once(attr, echo::cache_op_kernel,
                              (3 * kSlotCacheMax + 2 * kEntCacheMax) * static_cast<int>(sizeof(int32_t)),
                              "cache-manager smem attribute"))
    return r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(echo::kCoopThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(3 * P.slot_cache_cap + 2 * P.ent_cache_cap) * sizeof(int32_t);
  cfg.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, echo::cache_op_kernel, P);
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "cache-manager kernel");
}

int launch_pool_alloc(const echo_pool *pool, const echo_workspace *ws, const int32_t *host_idx, const int32_t *n_dev,
                      int32_t max_n, int32_t clock, const int32_t *clock_dev, int32_t *out_slots, int32_t *status,
                      cudaStream_t s) {
  echo::OpParams P = base_params(pool, ws, echo::kModeAlloc, clock, clock_dev, status);
  P.F = max_n;
  P.rows = host_idx;
  P.n_dev = n_dev;
  P.out_slots = out_slots;
  return run_op(P, s);
}

int launch_pool_evict(const echo_pool *pool, const echo_workspace *ws, const int32_t *n_needed_dev, int32_t clock,
                      const int32_t *clock_dev, int32_t *status, cudaStream_t s) {
  echo::OpParams P = base_params(pool, ws, echo::kModeEvict, clock, clock_dev, status);
  P.evict_n_dev = n_needed_dev;
  return run_op(P, s);
}

int launch_recall(const echo_pool *pool, const echo_workspace *ws, const int32_t *sel, const int32_t *req_to_host,
                  const int32_t *ctx_len, int B, int n_q, int k, int L_max, const echo_stage *stage, int32_t clock,
                  const int32_t *clock_dev, int32_t *out_slot, echo_stats *stats, int32_t *status, cudaStream_t s,
                  float *ema_s_hat, const float *ema_kth, int ema_n, float ema_alpha, int32_t *clock_advance,
                  int claimed) {
  echo::OpParams P = base_params(pool, ws, echo::kModeRecall, clock, clock_dev, status);
  P.claimed = claimed;
  P.F = B * n_q * k;
  P.sel = sel;
  P.req_to_host = req_to_host;
  P.n_q = n_q;
  P.k = k;
  P.L_max = L_max;
  P.B = B;
  P.ctx_len = ctx_len;
  P.stats = stats;
  P.out_slot = out_slot;
  if (stage && stage->reserve) {  // direct to slot
    P.reserve = stage->reserve;
    P.reserve_ctl = stage->reserve_ctl;
    P.reserve_cap = stage->reserve_cap;
  } else if (stage) {
    P.stage_host = stage->host_row;
    P.stage_count = stage->count;
    P.stage_rows = stage->rows;
    P.stage_stride = stage->stride;
    P.cap_div = stage->cap_div;
  }
  P.s_hat = ema_s_hat;
  P.kth = ema_kth;
  P.n_ema = ema_s_hat ? ema_n : 0;
  P.alpha = ema_alpha;
  P.clock_advance = clock_advance;
  return run_op(P, s, claimed != 0);  // after the decode step's top-k: programmatic launch
}

// the probe's grid barrier counts in words of its own, set back to zero before each
// probe (a barrier that gave up leaves its arrival count short of the grid)
static __device__ uint32_t g_probe_barrier[echo::kGCount];

int launch_wait_probe(int which, int32_t *status, cudaStream_t s) {
  uint32_t *glob = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&glob), g_probe_barrier);
  if (e != cudaSuccess) return cuda_fail(e, "wait probe scratch");
  if (which == 0) {
    echo::wait_probe_kernel<<<1, echo::kCoopThreads, 0, s>>>(0, glob, status);
    return check("wait probe");
  }
  e = cudaMemsetAsync(glob, 0, sizeof(g_probe_barrier), s);
  if (e != cudaSuccess) return cuda_fail(e, "wait probe reset");
  const int grid = sm_count() < 8 ? sm_count() : 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(echo::kCoopThreads);
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, echo::wait_probe_kernel, 1, glob, status);
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "wait probe");
}

int launch_append(const echo_pool *pool, const echo_workspace *ws, uint8_t *k_index, int32_t *ctx_len,
                  const int32_t *req_to_host, int B, int L_max, const uint16_t *new_kv, const uint8_t *new_k_index,
                  int32_t clock, const int32_t *clock_dev, echo_stats *stats, int32_t *status, cudaStream_t s) {
  if (B == 0) return ECHO_OK;
  echo::OpParams P = base_params(pool, ws, echo::kModeAppend, clock, clock_dev, status);
  P.F = B;
  P.rows = P.ws.entry_rows;
  P.new_kv = new_kv;
  P.stats = stats;
  echo::append_prepare_kernel<<<B, 128, 0, s>>>(P.pool, P.ws, k_index, ctx_len, req_to_host, B, L_max, new_kv,
                                                 new_k_index, status);
  int r = check("append prepare");
  if (r) return r;
  return run_op(P, s);
}

// ---------------------------------------------------------------------------
// scratch for callers that cannot allocate (echo_prefetch_recall_noalloc)
// ---------------------------------------------------------------------------
// One fixed array per device for the whole process: the recall's workspace laid
// out for at most kNoAllocMaxSlots GPU-pool slots and kNoAllocMaxRows selected
// entries.  It is shared by every call, so calls that overlap on the GPU race.
constexpr int32_t kNoAllocMaxSlots = 262144;
constexpr int32_t kNoAllocMaxRows = 32768;
constexpr size_t kNoAllocBytes = 4u << 20;  // >= the layout of the two maxima (checked below)
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// Device address of the array on the current device.  Host code cannot use the
// symbol itself as an address, so the address is looked up with that device
// current: on every call made outside stream capture (a context re-created after
// cudaDeviceReset gets its own address), and kept per device for calls made while
// the stream is capturing, which may not make the lookup.
static std::atomic<void *> g_noalloc_addr[kMaxDevices];

int noalloc_workspace(int32_t n_g, int32_t rows, cudaStream_t stream, echo_workspace *out) {
  if (workspace_bytes(kNoAllocMaxSlots, kNoAllocMaxRows) > kNoAllocBytes) {
    set_error("no-allocation scratch too small for its stated maxima");
    return ECHO_ENOTSUP;
  }
  if (n_g > kNoAllocMaxSlots || rows > kNoAllocMaxRows) {
    set_error("no-allocation recall supports pools of at most %d slots and at most %d selected entries "
              "(got %d slots, %d entries); use echo_prefetch_recall with a caller workspace",
              kNoAllocMaxSlots, kNoAllocMaxRows, n_g, rows);
    return ECHO_EINVAL;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device index %d out of range (the library serves devices 0..%d)", dev, kMaxDevices - 1);
    return ECHO_ENOTSUP;
  }
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
  void *p = nullptr;
  if (cs == cudaStreamCaptureStatusNone) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the no-allocation scratch");
    g_noalloc_addr[dev].store(p, std::memory_order_release);
  } else {
    p = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!p) {
      set_error("echo_prefetch_recall_noalloc: the first call on device %d must come before stream capture", dev);
      return ECHO_EINVAL;
    }
  }
  out->base = p;
  out->bytes = kNoAllocBytes;
  out->n_g = n_g;
  out->max_rows = rows;
  return ECHO_OK;
}

int launch_ema(float *s_hat, const float *kth, int n, int stride, float alpha, cudaStream_t s) {
  echo::ema_kernel<<<(n + 255) / 256, 256, 0, s>>>(s_hat, kth, n, stride, alpha);
  return check("ema");
}

}  // namespace echo_host
