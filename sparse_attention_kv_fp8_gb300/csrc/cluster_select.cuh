// cluster_select.cuh -- building blocks of the exact selections done by one
// thread-block cluster whose CTAs each hold a slice of the keys in shared memory
// (the top-k of a score row; the arg-top-k of the lowest eviction priorities):
//   - block and cluster prefix scans of two counters,
//   - cluster min / max of the keys,
//   - one radix step: per-CTA histogram of a digit (warp-aggregated atomics, so
//     runs of equal digits do not serialise), cluster-wide reduction through
//     distributed shared memory, and the digit where the running count reaches
//     the requested rank.
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

struct alignas(16) SelSmem {
  uint32_t hist[kMaxBins];
  uint32_t tot[kMaxBins];
  uint32_t wa[kSelWarps], wb[kSelWarps];
  uint32_t pub[4];      // values this CTA publishes to the cluster
  uint32_t result[2];   // digit, count before it
};

// exclusive block scan of two counters; block totals in ta / tb
__device__ __forceinline__ void sel_block_scan2(uint32_t a, uint32_t b, uint32_t &ea, uint32_t &eb, uint32_t &ta,
                                                uint32_t &tb, SelSmem *S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) {
    S->wa[warp] = ia;
    S->wb[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t x = S->wa[lane], y = S->wb[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t xa = __shfl_up_sync(0xffffffffu, x, o), xb = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += xa;
        y += xb;
      }
    }
    S->wa[lane] = x;
    S->wb[lane] = y;
  }
  __syncthreads();
  ea = (warp ? S->wa[warp - 1] : 0) + ia - a;
  eb = (warp ? S->wb[warp - 1] : 0) + ib - b;
  ta = S->wa[kSelWarps - 1];
  tb = S->wb[kSelWarps - 1];
  __syncthreads();
}

// every CTA publishes (a, b); returns the sums over lower ranks and over all ranks
__device__ __forceinline__ void sel_cluster_prefix2(cg::cluster_group &cl, SelSmem *S, uint32_t a, uint32_t b,
                                                    uint32_t &pa, uint32_t &pb, uint32_t &ga, uint32_t &gb) {
  if (threadIdx.x == 0) {
    S->pub[0] = a;
    S->pub[1] = b;
  }
  cl.sync();
  const int rank = static_cast<int>(cl.block_rank()), C = static_cast<int>(cl.num_blocks());
  pa = pb = ga = gb = 0;
  for (int r = 0; r < C; ++r) {
    const SelSmem *R = cl.map_shared_rank(S, r);
    const uint32_t x = R->pub[0], y = R->pub[1];
    if (r < rank) {
      pa += x;
      pb += y;
    }
    ga += x;
    gb += y;
  }
  cl.sync();
}

// cluster-wide min and max of per-thread values
__device__ __forceinline__ void sel_cluster_minmax(cg::cluster_group &cl, SelSmem *S, uint32_t mn, uint32_t mx,
                                                   uint32_t &gmn, uint32_t &gmx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  if (lane == 0) {
    S->wa[warp] = mn;
    S->wb[warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = S->wa[0], b = S->wb[0];
    for (int w = 1; w < kSelWarps; ++w) {
      a = min(a, S->wa[w]);
      b = max(b, S->wb[w]);
    }
    S->pub[2] = a;
    S->pub[3] = b;
  }
  cl.sync();
  const int C = static_cast<int>(cl.num_blocks());
  gmn = 0xFFFFFFFFu;
  gmx = 0;
  for (int r = 0; r < C; ++r) {
    const SelSmem *R = cl.map_shared_rank(S, r);
    gmn = min(gmn, R->pub[2]);
    gmx = max(gmx, R->pub[3]);
  }
  cl.sync();
}

// Histogram of digit `(x >> shift) & (nb - 1)` over the slice's reduced keys x whose
// bits above `hi` equal `prefix` (x >> hi == prefix >> hi).  `get(i, x)` returns
// false for slots that do not take part.  Equal digits within a warp are merged
// into one atomic.
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
    const uint32_t bin = act ? (x >> shift) & static_cast<uint32_t>(nb - 1) : 0xFFFFFFFFu;
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (act && lane == __ffs(peers) - 1) atomicAdd(&S->hist[bin], static_cast<uint32_t>(__popc(peers)));
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
  for (int i = threadIdx.x; i < nb; i += kSelThreads) {
    uint32_t s = 0;
    for (int r = 0; r < C; ++r) s += cl.map_shared_rank(S->hist, r)[i];
    S->tot[i] = s;
  }
  __syncthreads();
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
  cl.sync();  // remote reads of the histograms done before any CTA reuses them
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
