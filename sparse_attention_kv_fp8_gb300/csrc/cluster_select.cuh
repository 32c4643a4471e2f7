// cluster_select.cuh -- building blocks of the exact selections done by one
// thread-block cluster whose CTAs each hold a slice of the keys in shared memory
// (the top-k of a score row; the arg-top-k of the lowest eviction priorities):
//   - block and cluster prefix scans of two counters,
//   - cluster min / max of the keys,
//   - one radix step: per-CTA histogram of a digit (one atomic per warp when the
//     warp's digits agree), cluster-wide reduction through distributed shared
//     memory (each CTA owns a slice of the bins; remote loads are issued together,
//     never one after another), and the digit where the running count reaches the
//     requested rank.
// Keys are reduced to (key - min) first, so the digits cover only the bits in
// which the keys differ (priority clocks usually span a few bits, fp32 scores of
// one row about 25).
#pragma once

#include <cooperative_groups.h>

#include "echo_common.cuh"

namespace echo {

namespace cg = cooperative_groups;

constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kDigitBits = 12;
constexpr int kMaxBins = 1 << kDigitBits;

constexpr int kScanVals = 4;  // counters a scan carries at most

// The two halves of a cluster barrier (every thread of every CTA of the cluster
// executes each once per barrier): arrive when this thread's last read of another
// CTA's shared memory is done, wait before the shared memory may go away.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

struct alignas(16) SelSmem {
  uint32_t hist[kMaxBins];
  uint32_t tot[kMaxBins];
  uint32_t ws[kScanVals][kSelWarps];  // per-warp partial sums of a block scan
  uint32_t pub[8];                    // values this CTA publishes to the cluster
  uint32_t res[2 * kScanVals];        // results handed from warp 0 to the block
  uint32_t result[2];                 // digit, count before it
};

// exclusive block scan of NV counters; block totals in tot
template <int NV>
__device__ __forceinline__ void sel_block_scan(const uint32_t (&v)[NV], uint32_t (&ex)[NV], uint32_t (&tot)[NV],
                                               SelSmem *S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) inc[k] = v[k];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, inc[k], o);
      if (lane >= o) inc[k] += u;
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int k = 0; k < NV; ++k) S->ws[k][warp] = inc[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      uint32_t x = S->ws[k][lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      S->ws[k][lane] = x;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    ex[k] = (warp ? S->ws[k][warp - 1] : 0) + inc[k] - v[k];
    tot[k] = S->ws[k][kSelWarps - 1];
  }
  __syncthreads();
}

// exclusive block scan of two counters; block totals in ta / tb
__device__ __forceinline__ void sel_block_scan2(uint32_t a, uint32_t b, uint32_t &ea, uint32_t &eb, uint32_t &ta,
                                                uint32_t &tb, SelSmem *S) {
  const uint32_t v[2] = {a, b};
  uint32_t e[2], t[2];
  sel_block_scan<2>(v, e, t, S);
  ea = e[0];
  eb = e[1];
  ta = t[0];
  tb = t[1];
}

constexpr int kMaxCluster = 16;

// every CTA publishes NV counters; returns their sums over lower ranks (pre) and
// over all ranks (all).  Warp 0 reads the C published vectors (one remote load per
// lane and counter, all in flight at once), scans them, and hands the result to the
// block through shared memory.
template <int NV>
__device__ __forceinline__ void sel_cluster_prefix(cg::cluster_group &cl, SelSmem *S, const uint32_t (&mine)[NV],
                                                   uint32_t (&pre)[NV], uint32_t (&all)[NV]) {
  if (threadIdx.x == 0) {
#pragma unroll
    for (int k = 0; k < NV; ++k) S->pub[k] = mine[k];
  }
  cl.sync();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int rank = static_cast<int>(cl.block_rank()), C = static_cast<int>(cl.num_blocks());
    uint32_t x[NV];
    const SelSmem *R = cl.map_shared_rank(S, lane < C ? lane : 0);
#pragma unroll
    for (int k = 0; k < NV; ++k) x[k] = lane < C ? R->pub[k] : 0u;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      uint32_t sx = x[k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, sx, o);
        if (lane >= o) sx += u;
      }
      const uint32_t e = __shfl_sync(0xffffffffu, sx - x[k], rank);
      const uint32_t t = __shfl_sync(0xffffffffu, sx, 31);
      if (lane == 0) {
        S->res[k] = e;
        S->res[kScanVals + k] = t;
      }
    }
  }
  cl.sync();  // also orders the remote reads above before any CTA republishes
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    pre[k] = S->res[k];
    all[k] = S->res[kScanVals + k];
  }
  __syncthreads();
}

__device__ __forceinline__ void sel_cluster_prefix2(cg::cluster_group &cl, SelSmem *S, uint32_t a, uint32_t b,
                                                    uint32_t &pa, uint32_t &pb, uint32_t &ga, uint32_t &gb) {
  const uint32_t m[2] = {a, b};
  uint32_t p[2], g[2];
  sel_cluster_prefix<2>(cl, S, m, p, g);
  pa = p[0];
  pb = p[1];
  ga = g[0];
  gb = g[1];
}

// cluster-wide min and max of per-thread values (at most once per launch: the
// published pair is not overwritten afterwards, so remote readers need no second barrier)
__device__ __forceinline__ void sel_cluster_minmax(cg::cluster_group &cl, SelSmem *S, uint32_t mn, uint32_t mx,
                                                   uint32_t &gmn, uint32_t &gmx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    S->ws[0][warp] = mn;
    S->ws[1][warp] = mx;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t a = S->ws[0][lane], b = S->ws[1][lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      S->pub[4] = a;
      S->pub[5] = b;
    }
  }
  cl.sync();
  if (warp == 0) {
    const int C = static_cast<int>(cl.num_blocks());
    const SelSmem *R = cl.map_shared_rank(S, lane < C ? lane : 0);
    uint32_t a = lane < C ? R->pub[4] : 0xFFFFFFFFu;
    uint32_t b = lane < C ? R->pub[5] : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
      b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
    }
    if (lane == 0) {
      S->res[0] = a;
      S->res[1] = b;
    }
  }
  __syncthreads();  // pub[4..5] are written once per launch: no second cluster barrier
  gmn = S->res[0];
  gmx = S->res[1];
  __syncthreads();
}

// Histogram of digit `(x >> shift) & (nb - 1)` over the slice's reduced keys x whose
// bits above `hi` equal `prefix` (x >> hi == prefix >> hi).  `get(i, x)` returns
// false for slots that do not take part.  A warp whose taking-part lanes all hold
// one digit adds once; otherwise each lane adds its own (bank-parallel).
template <typename Get>
__device__ __forceinline__ void sel_histogram(SelSmem *S, int n, int hi, int shift, int nb, uint32_t prefix,
                                              Get get) {
  for (int i = threadIdx.x; i < nb; i += kSelThreads) S->hist[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  for (int base = (threadIdx.x & ~31); base < n; base += kSelThreads) {
    const int i = base + lane;
    uint32_t x = 0;
    bool act = i < n && get(i, x);
    if (act && hi < 32) act = (x >> hi) == (prefix >> hi);
    const uint32_t bin = (x >> shift) & static_cast<uint32_t>(nb - 1);
    const uint32_t am = __ballot_sync(0xffffffffu, act);
    if (am == 0) continue;
    const int first = __ffs(am) - 1;
    const uint32_t b0 = __shfl_sync(0xffffffffu, bin, first);
    if (__all_sync(0xffffffffu, !act || bin == b0)) {
      if (lane == first) atomicAdd(&S->hist[b0], static_cast<uint32_t>(__popc(am)));
    } else if (act) {
      atomicAdd(&S->hist[bin], 1u);
    }
  }
  __syncthreads();
}

// The digit at which the cluster-wide count, taken from the top digit down
// (descending) or from 0 up, first reaches `need` (>= 1), and the count strictly
// before it.  Every CTA gets the same answer.
__device__ __forceinline__ void sel_find_digit(cg::cluster_group &cl, SelSmem *S, int nb, uint32_t need,
                                               bool descending, uint32_t &digit, uint32_t &before) {
  cl.sync();  // every slice histogram complete
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  // 1. CTA `rank` owns bins [o0, o1) and sums them over the cluster (remote loads in flight together)
  const int per_owner = (nb + C - 1) / C;
  const int o0 = rank * per_owner < nb ? rank * per_owner : nb;
  const int o1 = o0 + per_owner < nb ? o0 + per_owner : nb;
  for (int i = o0 + static_cast<int>(threadIdx.x); i < o1; i += kSelThreads) {
    uint32_t v[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) v[r] = r < C ? cl.map_shared_rank(S->hist, r)[i] : 0u;
    uint32_t s = 0;
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) s += v[r];
    S->tot[i] = s;
  }
  cl.sync();  // owners' totals complete
  // 2. gather every owner's totals (rows of another owner are read remotely)
  for (int i = threadIdx.x; i < nb; i += kSelThreads) {
    const int owner = i / per_owner;
    if (owner != rank) S->tot[i] = cl.map_shared_rank(S->tot, owner)[i];
  }
  __syncthreads();
  // 3. running count in the requested direction; the digit where it reaches `need`
  const int per = (nb + kSelThreads - 1) / kSelThreads;
  const int p0 = threadIdx.x * per;
  uint32_t c = 0;
  for (int u = 0; u < per; ++u) {
    const int idx = p0 + u;
    if (idx < nb) c += S->tot[descending ? nb - 1 - idx : idx];
  }
  uint32_t ex, dz, tt, tz;
  sel_block_scan2(c, 0, ex, dz, tt, tz, S);
  uint32_t run = ex;
  for (int u = 0; u < per; ++u) {
    const int idx = p0 + u;
    if (idx >= nb) break;
    const int bin = descending ? nb - 1 - idx : idx;
    const uint32_t cnt = S->tot[bin];
    if (run < need && run + cnt >= need) {
      S->result[0] = static_cast<uint32_t>(bin);
      S->result[1] = run;
    }
    run += cnt;
  }
  __syncthreads();
  digit = S->result[0];
  before = S->result[1];
  cl.sync();  // remote reads of the histograms and totals done before any CTA reuses them
}

// Exact selection of the need-th key (1-based) in the given direction among the
// cluster's reduced keys x = key - kmin (kmin, kmax the cluster min / max of the
// taking-part keys).  Returns the key T and how many keys equal to T are taken.
template <typename Get>
__device__ __forceinline__ void sel_radix_select(cg::cluster_group &cl, SelSmem *S, int n, uint32_t kmin,
                                                 uint32_t kmax, uint32_t need, bool descending, Get get, uint32_t &T,
                                                 uint32_t &need_eq) {
  const uint32_t range = kmax - kmin;
  int hi = range == 0 ? 0 : 32 - __clz(range);  // bits in which the reduced keys differ
  uint32_t prefix = 0;
  int pass_no = 0;
  (void)pass_no;
  while (hi > 0) {
    const int width = hi < kDigitBits ? hi : kDigitBits;
    const int shift = hi - width;
    const int nb = 1 << width;
    sel_histogram(S, n, hi, shift, nb, prefix, [&](int i, uint32_t &x) {
      uint32_t key;
      if (!get(i, key)) return false;
      x = key - kmin;
      return true;
    });
    ECHO_TRACE_MARK(16 + 2 * (pass_no & 3));
    uint32_t d, before;
    sel_find_digit(cl, S, nb, need, descending, d, before);
    ECHO_TRACE_MARK(17 + 2 * (pass_no & 3));
    ++pass_no;
    prefix |= d << shift;
    need -= before;
    hi = shift;
  }
  T = kmin + prefix;
  need_eq = need;
}

}  // namespace echo
