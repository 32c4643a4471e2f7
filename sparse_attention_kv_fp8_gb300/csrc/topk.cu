// topk.cu -- exact top-k of the index scores (ECHO review, marsggbo.github.io,
// "OSDI'26 | ECHO", section 2: the indexer scores every cached token and the k
// highest (k = 2048 in DeepSeek-V3.2) go to the sparse MLA; section 6.2 names
// radix select over the score bits as the selection machinery).
//
// sm_103a design: one thread-block cluster of kTopkCluster CTAs per (request,
// query) row (4 or 2 CTAs when the rows are many: see the launcher).  Each
// CTA keeps its slice of the row in shared memory as order-preserving uint32 keys (one
// global read).  The keys are reduced to
// key - min (cluster min / max), and a 12-bit digit of the reduced key (the top
// bits in which the row's keys differ) is histogrammed per CTA.  The cluster finds
// the digit d holding the target-th largest key in two small gathers over
// distributed shared memory: 64-bin coarse histograms first, then the 64 fine bins
// of the chosen coarse bin -- a few KB per CTA instead of whole histograms.  Every
// CTA then collects the keys of bin d from the whole cluster (usually a few dozen)
// and resolves the exact k-th key T and its own output offsets by itself.  A final
// pass writes the selected indices in ascending order (ties at T go to the lower
// index).  In the decode step the same kernel makes the recall's claims for the
// entries it selects, one entry per thread from a compacted list, with the
// request's host rows staged in shared memory before the scores are ready.
// A threshold bin with more than kCand keys falls back to full radix passes.
//
// In the decode step the indexer has already made the first radix step: it counts
// every score of the row in a kSelBins-bin histogram over a window of score keys
// this kernel chose from the row's previous step (just below the k-th key up to the
// largest).  The threshold bin then comes from that histogram directly -- no min /
// max round, no local histogram, no coarse / fine gathers -- and the keys of that bin
// are resolved as above.  Any window is exact (the bins are ordered like the keys);
// when it misses (fewer keys in it than k, or its threshold bin too full) the kernel
// takes the path above instead.
#include "cache_common.cuh"
#include "cluster_select.cuh"

ECHO_TRACE_UNIT(topk)

namespace echo {

constexpr int kTopkCluster = 8;
constexpr int kMaxChunk = 44 * 1024;  // keys per CTA kept in shared memory
constexpr int kCand = 1024;           // threshold-bin keys resolved without more radix passes
constexpr int kCoarse = 64;           // fine bins per coarse bin
constexpr int kCoarseBins = kMaxBins / kCoarse;
constexpr int kList = kMaxBins / 2;   // selected entries a CTA can list for the claims
constexpr int kTopkSmemMax = 232448;

struct alignas(16) TopkExtra {
  uint32_t cand_key[kCand];          // this CTA's keys in the threshold bin (read by the cluster)
  uint32_t all_key[kCand];           // the threshold-bin keys of the whole cluster, in rank order
  uint32_t coarse[kCoarseBins];      // this CTA's coarse histogram (read by the cluster)
  uint32_t ctot[kCoarseBins];        // cluster totals of the coarse bins
  uint32_t ftot[kCoarse];            // cluster totals of the fine bins of the chosen coarse bin
  uint32_t off[kMaxCluster + 1];     // offsets of each rank's candidates in all_key
  uint32_t cand_n, above;            // published: keys in the threshold bin, keys above it
  uint32_t kmax_pub;                 // published: this CTA's largest key (histogram path)
  uint32_t v[12];                    // block-wide values
  uint32_t hv[4];                    // histogram path: threshold bin, keys above it, keys in it, row max
};

// The bin at which the running count of 64 bins, taken from the highest bin down,
// reaches `need` (warp 0 only; cnt(i) gives the count of bin i, 0 <= i < 64).
// Writes the bin and the count above it to out[0], out[1].
template <typename Cnt>
__device__ __forceinline__ void warp_find_from_top64(uint32_t need, Cnt cnt, uint32_t *out) {
  const int lane = threadIdx.x & 31;
  const int b0 = 63 - 2 * lane, b1 = 62 - 2 * lane;
  const uint32_t c0 = cnt(b0), c1 = cnt(b1);
  const uint32_t s = c0 + c1;
  uint32_t inc = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  const uint32_t ex = inc - s;
  if (ex < need && need <= ex + c0) {
    out[0] = static_cast<uint32_t>(b0);
    out[1] = ex;
  } else if (ex + c0 < need && need <= ex + s) {
    out[0] = static_cast<uint32_t>(b1);
    out[1] = ex + c0;
  }
}

__global__ void __launch_bounds__(kSelThreads, 1)
    topk_kernel(const float *__restrict__ scores, const int32_t *__restrict__ ctx_len, int n_q, int L_max, int k,
                int chunk, int32_t *__restrict__ sel, float *__restrict__ kth, const ClaimArgs ca, int do_claim,
                int stage_r2h) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int row = blockIdx.x / C;
  const int b = row / n_q, j = row % n_q;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem *S = reinterpret_cast<SelSmem *>(smem_raw);
  TopkExtra *X = reinterpret_cast<TopkExtra *>(smem_raw + sizeof(SelSmem));
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem) + sizeof(TopkExtra));
  const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys);
  int32_t *r2s = reinterpret_cast<int32_t *>(keys + chunk);  // staged host rows (stage_r2h)
  uint32_t *list_pos = S->tot, *list_tok = S->tot + kList;   // claim list (tot is free by then)
  ECHO_TRACE_FIRST(24);

  // ---- what does not come from the kernel before: the row's length, its host rows,
  // the step clock
  int L = __ldg(ctx_len + b);
  L = L < 0 ? 0 : (L > L_max ? L_max : L);
  const int Lr = query_valid_len(L, n_q, j);
  const int target = Lr < k ? Lr : k;
  const int lo = rank * chunk;
  const int hi = lo + chunk < Lr ? lo + chunk : Lr;
  const int n_local = hi > lo ? hi - lo : 0;
  const int32_t *r2h = do_claim ? ca.req_to_host + static_cast<size_t>(b) * L_max + lo : nullptr;
  const int32_t clock = do_claim ? (ca.clock_dev ? *ca.clock_dev : ca.clock) : 0;
  if (stage_r2h)
    for (int i = threadIdx.x; i < n_local; i += kSelThreads) r2s[i] = __ldg(r2h + i);
  for (int i = threadIdx.x; i < kCoarseBins; i += kSelThreads) X->ctot[i] = 0;
  if (threadIdx.x < kCoarse) X->ftot[threadIdx.x] = 0;
  if (threadIdx.x < 12) X->v[threadIdx.x] = 0;
  if (threadIdx.x < 4) X->hv[threadIdx.x] = 0;
  // decode step: the histogram of this row's scores the indexer made over the key
  // window the last step chose (written by this kernel's previous launch, so it is
  // read before the programmatic wait)
  int4 hint = make_int4(0, 0, 0, 0);
  if (do_claim && row < kSelHintRows) hint = ca.ws.sel_hint[row];
  const uint32_t *hist_row = hint.z ? ca.ws.sel_hist + static_cast<size_t>(row) * kSelBins : nullptr;
  const uint32_t hlo = static_cast<uint32_t>(hint.x), hsh = static_cast<uint32_t>(hint.y);

  pdl_wait();  // the scores come from the kernel before (programmatic launch)
  pdl_launch_dependents();
  // this thread's two bins of the histogram (highest first), loaded while the keys load
  uint32_t hc0 = 0, hc1 = 0;
  if (hist_row && target > 0) {
    hc0 = __ldcg(hist_row + (kSelBins - 1 - 2 * static_cast<int>(threadIdx.x)));
    hc1 = __ldcg(hist_row + (kSelBins - 2 - 2 * static_cast<int>(threadIdx.x)));
  }
  ECHO_TRACE_FIRST(26);
  ECHO_TRACE_MARK(0);
  const float *srow = scores + static_cast<size_t>(row) * L_max;
  int32_t *out = sel + static_cast<size_t>(row) * k;

  // ---- the slice as order-preserving keys (16-byte loads when aligned), with its min / max
  uint32_t mn = 0xFFFFFFFFu, mx = 0;
  if ((reinterpret_cast<uintptr_t>(srow + lo) & 15) == 0) {
    const int nv = n_local >> 2;
    const float4 *src = reinterpret_cast<const float4 *>(srow + lo);
    for (int i = threadIdx.x; i < nv; i += kSelThreads) {
      const float4 v = __ldcg(src + i);
      const uint32_t a = score_key(v.x), b2 = score_key(v.y), c = score_key(v.z), d = score_key(v.w);
      reinterpret_cast<uint4 *>(keys)[i] = make_uint4(a, b2, c, d);
      mn = min(min(mn, a), min(b2, min(c, d)));
      mx = max(max(mx, a), max(b2, max(c, d)));
    }
    for (int i = (nv << 2) + threadIdx.x; i < n_local; i += kSelThreads) {
      const uint32_t a = score_key(__ldcg(srow + lo + i));
      keys[i] = a;
      mn = min(mn, a);
      mx = max(mx, a);
    }
  } else {
    for (int i = threadIdx.x; i < n_local; i += kSelThreads) {
      const uint32_t a = score_key(__ldcg(srow + lo + i));
      keys[i] = a;
      mn = min(mn, a);
      mx = max(mx, a);
    }
  }
  // this thread's segment of the slice: [s0, s1), read as 16-byte vectors
  int seg = (n_local + kSelThreads - 1) / kSelThreads;
  seg = (seg + 3) & ~3;
  const int s0 = threadIdx.x * seg < n_local ? threadIdx.x * seg : n_local;
  const int s1 = s0 + seg < n_local ? s0 + seg : n_local;
  __syncthreads();
  ECHO_TRACE_MARK(1);

  // ---- the target-th largest key T, how many keys equal to T are taken (needT), and
  // this CTA's output offsets (keys above T and equal to T in lower CTAs)
  uint32_t T = 0, needT = 0, pg = 0, pe = 0;
  uint32_t row_max = 0;  // the row's largest key (for the next step's histogram window)
  bool offsets_known = false;
  // candidate path: bit j of this thread's segment lies above the threshold bin
  // (selected whatever T is) / in it; thr_above counts the first kind
  const bool masks = s1 - s0 <= 64;
  uint64_t above_mask = 0, cand_mask = 0;
  uint32_t thr_above = 0;
  bool classified = false;  // the candidate path filled the masks above
  bool arrived = false;  // this CTA has made its last remote shared-memory read
  if (target > 0) {
    // (1) the indexer's histogram: the bin d where the count from the top bin down
    // reaches the target.  Every CTA reads the same counts, so every CTA takes the
    // same branch; a window that misses (fewer keys in it than the target, or a
    // threshold bin too full to resolve directly) falls back to (2).
    bool fast = false;
    if (hist_row) {
      static_assert(kSelBins == 2 * kSelThreads, "two histogram bins per thread");
      uint32_t ex, dz, tot, tz;
      sel_block_scan2(hc0 + hc1, 0u, ex, dz, tot, tz, S);
      const uint32_t tgt = static_cast<uint32_t>(target);
      if (ex < tgt && tgt <= ex + hc0) {
        X->hv[0] = kSelBins - 1 - 2 * threadIdx.x;
        X->hv[1] = ex;
        X->hv[2] = hc0;
      } else if (ex + hc0 < tgt && tgt <= ex + hc0 + hc1) {
        X->hv[0] = kSelBins - 2 - 2 * threadIdx.x;
        X->hv[1] = ex + hc0;
        X->hv[2] = hc1;
      }
      __syncthreads();
      fast = tot >= tgt && X->hv[2] <= static_cast<uint32_t>(kCand);
    }
    uint32_t kmin = 0, kmax = 0, d = 0, above_d = 0, cnt_d = 0;
    int shift = 0;
    if (fast) {
      d = X->hv[0];
      above_d = X->hv[1];
      cnt_d = X->hv[2];
    } else {
    // (2) cluster min / max, a 12-bit digit of key - min, coarse and fine bins
    sel_cluster_minmax(cl, S, mn, mx, kmin, kmax);
    row_max = kmax;
    ECHO_TRACE_MARK(2);
    const uint32_t range = kmax - kmin;
    const int hb = range == 0 ? 0 : 32 - __clz(range);
    const int width = hb < kDigitBits ? hb : kDigitBits;
    shift = hb - width;
    const int nb = 1 << width;
    const int nco = (nb + kCoarse - 1) / kCoarse;
    // fine histogram of the digit (key - kmin) >> shift, one shared-memory atomic per key
    for (int i = threadIdx.x; i < nb; i += kSelThreads) S->hist[i] = 0;
    __syncthreads();
    if (nb == 1) {
      if (threadIdx.x == 0) S->hist[0] = static_cast<uint32_t>(n_local);
    } else {
      for (int i = s0; i < s1; i += 4) {
        const uint4 v = keys4[i >> 2];
        atomicAdd(&S->hist[(v.x - kmin) >> shift], 1u);
        if (i + 1 < s1) atomicAdd(&S->hist[(v.y - kmin) >> shift], 1u);
        if (i + 2 < s1) atomicAdd(&S->hist[(v.z - kmin) >> shift], 1u);
        if (i + 3 < s1) atomicAdd(&S->hist[(v.w - kmin) >> shift], 1u);
      }
    }
    __syncthreads();
    // coarse histogram: one warp per coarse bin
    for (int cb = warp; cb < nco; cb += kSelWarps) {
      uint32_t c = 0;
      for (int i = lane; i < kCoarse; i += 32) c += cb * kCoarse + i < nb ? S->hist[cb * kCoarse + i] : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) X->coarse[cb] = c;
    }
    cl.sync();  // every CTA's fine and coarse histograms complete
    ECHO_TRACE_MARK(3);
    // cluster totals of the coarse bins; the coarse bin D holding the target-th key
    if (threadIdx.x < C * nco) {
      const int r = threadIdx.x / nco, cb = threadIdx.x % nco;
      const uint32_t v = cl.map_shared_rank(X->coarse, r)[cb];
      if (v) atomicAdd(&X->ctot[cb], v);
    }
    __syncthreads();
    if (warp == 0)
      warp_find_from_top64(static_cast<uint32_t>(target), [&](int i) { return i < nco ? X->ctot[i] : 0u; },
                           &X->v[0]);
    __syncthreads();
    const uint32_t D = X->v[0], above_D = X->v[1];
    // cluster totals of D's fine bins; the digit d
    if (threadIdx.x < C * kCoarse) {
      const int r = threadIdx.x / kCoarse, i = threadIdx.x % kCoarse;
      const int fb = static_cast<int>(D) * kCoarse + i;
      if (fb < nb) {
        const uint32_t v = cl.map_shared_rank(S->hist, r)[fb];
        if (v) atomicAdd(&X->ftot[i], v);
      }
    }
    __syncthreads();
    if (warp == 0) {
      warp_find_from_top64(static_cast<uint32_t>(target) - above_D, [&](int i) { return X->ftot[i]; }, &X->v[2]);
      __syncwarp();
      // this CTA's keys above bin d: coarse bins above D, then D's fine bins above d
      const uint32_t dd = D * kCoarse + X->v[2];
      uint32_t a = 0;
      for (int cb = static_cast<int>(D) + 1 + lane; cb < nco; cb += 32) a += X->coarse[cb];
      for (int i = lane; i < kCoarse; i += 32) {
        const uint32_t fb = D * kCoarse + i;
        if (fb > dd && fb < static_cast<uint32_t>(nb)) a += S->hist[fb];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0) X->above = a;
    }
    __syncthreads();
    d = D * kCoarse + X->v[2];
    above_d = above_D + X->v[3];
    cnt_d = X->ftot[X->v[2]];
    }
    const uint32_t need_d = static_cast<uint32_t>(target) - above_d;
    ECHO_TRACE_VALUE(27, cnt_d);
    ECHO_TRACE_VALUE(28, (fast ? 1u : 0u) | (hist_row ? 2u : 0u));
    ECHO_TRACE_VALUE(29, hsh);
    ECHO_TRACE_VALUE(30, hlo);
    ECHO_TRACE_VALUE(31, d);
    // bin d as a key range [blo, bhi] in either form (the last histogram bin is open above)
    const unsigned long long base = fast ? hlo : kmin;
    const int bsh = fast ? static_cast<int>(hsh) : shift;
    const unsigned long long top = 0xFFFFFFFFull;
    const uint32_t blo = static_cast<uint32_t>(min(base + (static_cast<unsigned long long>(d) << bsh), top));
    const uint32_t bhi =
        (fast && d == kSelBins - 1)
            ? 0xFFFFFFFFu
            : static_cast<uint32_t>(min(base + (static_cast<unsigned long long>(d + 1) << bsh) - 1ull, top));
    ECHO_TRACE_MARK(4);
    if (cnt_d <= static_cast<uint32_t>(kCand)) {
      // publish this CTA's keys of bin d (and, histogram path, how many of its keys lie
      // above bin d and its largest key); every CTA collects the cluster's and resolves T
      {
        uint32_t c = 0, a = 0;
        for (int i = s0; i < s1; i += 4) {
          const uint4 v = keys4[i >> 2];
          const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (i + u < s1) {
              const bool above = kv[u] > bhi, in = !above && kv[u] >= blo;
              c += in;
              a += above;
              if (masks) {
                above_mask |= static_cast<uint64_t>(above) << (i + u - s0);
                cand_mask |= static_cast<uint64_t>(in) << (i + u - s0);
              }
            }
        }
        thr_above = a;
        classified = masks;
        if (c) {  // rare: a second pass over the segment writes them
          const uint32_t slot = atomicAdd(&X->v[5], c);
          for (int i = s0, q = 0; i < s1 && q < static_cast<int>(c); ++i) {
            const uint32_t key = keys[i];
            if (key >= blo && key <= bhi) X->cand_key[slot + q++] = key;
          }
        }
        if (fast) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          }
          if (lane == 0) {
            if (a) atomicAdd(&X->v[11], a);
            atomicMax(&X->hv[3], mx);
          }
        }
        __syncthreads();
        ECHO_TRACE_MARK(11);
        if (threadIdx.x == 0) {
          X->cand_n = X->v[5];
          if (fast) {
            X->above = X->v[11];
            X->kmax_pub = X->hv[3];
          }
        }
      }
      cl.sync();  // every CTA's candidates published
      ECHO_TRACE_MARK(12);
      if (warp == 0) {
        const TopkExtra *R = cl.map_shared_rank(X, lane < C ? lane : 0);
        const uint32_t n = lane < C ? R->cand_n : 0u, a = lane < C ? R->above : 0u;
        if (fast) {  // the row's largest key
          uint32_t m = lane < C ? R->kmax_pub : 0u;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
          if (lane == 0) X->hv[3] = m;
        }
        uint32_t inc = n, ia = a;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t u = __shfl_up_sync(0xffffffffu, inc, o);
          const uint32_t ua = __shfl_up_sync(0xffffffffu, ia, o);
          if (lane >= o) {
            inc += u;
            ia += ua;
          }
        }
        if (lane <= C) X->off[lane] = inc - n;  // lane C: the total
        if (lane == rank) X->v[6] = ia - a;     // keys above bin d in lower CTAs
      }
      __syncthreads();
      ECHO_TRACE_MARK(13);
      const int nc = static_cast<int>(X->off[C]);
      for (int g = threadIdx.x; g < nc; g += kSelThreads) {
        int r = 0;
        while (r + 1 < C && X->off[r + 1] <= static_cast<uint32_t>(g)) ++r;
        X->all_key[g] = cl.map_shared_rank(X->cand_key, r)[g - static_cast<int>(X->off[r])];
      }
      __syncthreads();
      // the last read of another CTA's shared memory on this path: arrive at the cluster
      // barrier that lets the CTAs exit, wait for it only at the end
      cluster_arrive();
      arrived = true;
      ECHO_TRACE_MARK(14);
      for (int i = threadIdx.x; i < nc; i += kSelThreads) {
        const uint32_t ki = X->all_key[i];
        uint32_t greater = 0, equal = 0;
        for (int jj = 0; jj < nc; ++jj) {
          const uint32_t kj = X->all_key[jj];
          greater += kj > ki;
          equal += kj == ki;
        }
        if (greater < need_d && need_d <= greater + equal) {  // every such thread holds the same key
          X->v[7] = ki;
          X->v[8] = need_d - greater;
        }
      }
      __syncthreads();
      ECHO_TRACE_MARK(15);
      T = X->v[7];
      needT = X->v[8];
      // lower CTAs' candidates above / equal to T (one warp-wide count per 32 candidates)
      const int n_lower = static_cast<int>(X->off[rank]);
      for (int base = warp * 32; base < n_lower; base += kSelThreads) {
        const int i = base + lane;
        const uint32_t ki = i < n_lower ? X->all_key[i] : 0u;
        const uint32_t gm = __ballot_sync(0xffffffffu, i < n_lower && ki > T);
        const uint32_t em = __ballot_sync(0xffffffffu, i < n_lower && ki == T);
        if (lane == 0) {
          if (gm) atomicAdd(&X->v[9], static_cast<uint32_t>(__popc(gm)));
          if (em) atomicAdd(&X->v[10], static_cast<uint32_t>(__popc(em)));
        }
      }
      __syncthreads();
      pg = X->v[6] + X->v[9];
      pe = X->v[10];
      offsets_known = true;
      if (fast) row_max = X->hv[3];
    } else if (shift == 0) {
      // every key of bin d equals T: counts of the histogram are exact
      T = kmin + d;
      needT = need_d;
      uint32_t ga, gb;
      sel_cluster_prefix2(cl, S, X->above, S->hist[d], pg, pe, ga, gb);
      offsets_known = true;
    } else {
      // many keys share the threshold bin (ties or a clustered row): exact radix passes
      cl.sync();  // no CTA still reads this CTA's histogram
      sel_radix_select(cl, S, n_local, kmin, kmax, static_cast<uint32_t>(target), true,
                       [&](int i, uint32_t &key) {
                         key = keys[i];
                         return true;
                       },
                       T, needT);
    }
  }
  ECHO_TRACE_MARK(5);

  // ---- ascending output: selected iff key > T, or key == T among the first needT
  // equal keys; each thread's segment is contiguous, so a block scan orders them
  uint32_t g = 0, e = 0;
  uint64_t sel_mask = 0;  // bit j: key s0 + j is above or equal to T (segments of at most 64)
  if (target > 0 && classified) {
    // the candidate path classified every key already: only the threshold bin's keys
    // (a handful per CTA) need comparing with T
    g = thr_above;
    sel_mask = above_mask;
    for (uint64_t m = cand_mask; m; m &= m - 1) {
      const int j = __ffsll(static_cast<long long>(m)) - 1;
      const uint32_t key = keys[s0 + j];
      g += key > T;
      e += key == T;
      if (key >= T) sel_mask |= 1ull << j;
    }
  } else if (target > 0)
    for (int i = s0; i < s1; i += 4) {
      const uint4 v = keys4[i >> 2];
      const uint32_t kv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + u < s1) {
          g += kv[u] > T;
          e += kv[u] == T;
          if (masks && kv[u] >= T) sel_mask |= 1ull << (i + u - s0);
        }
    }
  ECHO_TRACE_MARK(16);
  uint32_t eg, ee, tg, te;
  sel_block_scan2(g, e, eg, ee, tg, te, S);
  ECHO_TRACE_MARK(17);
  if (target > 0 && !offsets_known) {
    uint32_t gg, ge;
    sel_cluster_prefix2(cl, S, tg, te, pg, pe, gg, ge);
  }
  ECHO_TRACE_MARK(6);
  // the recall's claim of every selected entry (decode step): see cache_common.cuh
  const int f_row = row * k;
  const uint32_t mpe = pe < needT ? pe : needT;
  const uint32_t te_taken = (pe + te < needT ? pe + te : needT) - mpe;
  const uint32_t n_sel = target > 0 ? tg + te_taken : 0u;
  const bool use_list = do_claim && n_sel <= static_cast<uint32_t>(kList);
  // one compact pass over the keys at or above T only: positions, output, claim list
  if (target > 0 && (g | e)) {
    uint32_t gb = pg + eg, eb = pe + ee;
    uint64_t todo = masks ? sel_mask : ~0ull;
    for (int i = s0; i < s1 && todo; ++i) {
      if (masks) {
        i = s0 + __ffsll(static_cast<long long>(todo)) - 1;
        todo &= todo - 1;
      }
      const uint32_t key = keys[i];
      int pos = -1;
      uint32_t li = 0;
      if (key > T) {
        const uint32_t t_before = eb < needT ? eb : needT;
        li = (gb - pg) + (t_before - mpe);
        pos = static_cast<int>(gb + t_before);
        ++gb;
      } else if (key == T) {
        if (eb < needT) {
          li = (gb - pg) + (eb - mpe);
          pos = static_cast<int>(gb + eb);
        }
        ++eb;
      }
      if (pos < 0) continue;
      out[pos] = lo + i;
      if (use_list) {
        list_pos[li] = static_cast<uint32_t>(pos);
        list_tok[li] = static_cast<uint32_t>(i);
      }
    }
  }
  if (do_claim && !use_list && target > 0 && (g | e)) {
    // more selected entries in this CTA than the list holds: claim in a second pass
    uint32_t gb = pg + eg, eb = pe + ee;
    for (int i = s0; i < s1; ++i) {
      const uint32_t key = keys[i];
      int pos = -1;
      if (key > T) {
        pos = static_cast<int>(gb + (eb < needT ? eb : needT));
        ++gb;
      } else if (key == T) {
        if (eb < needT) pos = static_cast<int>(gb + eb);
        ++eb;
      }
      if (pos >= 0) claim_entry(ca.pool, ca.ws, f_row + pos, __ldg(r2h + i), clock, ca.status);
    }
  }
  ECHO_TRACE_MARK(8);
  if (use_list) {
    __syncthreads();
    ECHO_TRACE_MARK(9);
    for (int li = threadIdx.x; li < static_cast<int>(n_sel); li += kSelThreads) {
      const int i = static_cast<int>(list_tok[li]);
      const int32_t h = stage_r2h ? r2s[i] : __ldg(r2h + i);
      claim_entry(ca.pool, ca.ws, f_row + static_cast<int>(list_pos[li]), h, clock, ca.status);
    }
  }
  for (int i = target + rank * kSelThreads + threadIdx.x; i < k; i += C * kSelThreads) {
    out[i] = -1;
    if (do_claim) ca.ws.entry_h[f_row + i] = -1;
  }
  if (rank == 0 && threadIdx.x == 0) {
    kth[row] = target > 0 ? key_score(T) : -INFINITY;
    // the window of this row's histogram in the next step, in key space:
    // [T - max((max - T) / 4, 256), max], cut into kSelBins bins of 2^shift keys (keys
    // above it count in the last bin)
    if (do_claim && row < kSelHintRows) {
      int4 h = make_int4(0, 0, 0, 0);
      if (target > 0) {
        const uint32_t span = row_max - T;
        const uint32_t delta = max(span / 4u, 256u);
        const uint32_t lo = T > delta ? T - delta : 0u;
        const uint32_t width = row_max - lo;
        const int hb = 32 - __clz(width | 1u);
        h = make_int4(static_cast<int32_t>(lo), hb > kSelBinBits ? hb - kSelBinBits : 0, 1, 0);
      }
      ca.ws.sel_hint[row] = h;
    }
  }
  ECHO_TRACE_MARK(10);
  // no CTA leaves while others may still read its shared memory
  if (!arrived) cluster_arrive();
  cluster_wait();
  // every CTA of the cluster has read the histogram: back to zero for the next step
  if (hist_row)
    for (int i = rank * (kSelBins / C) + threadIdx.x; i < (rank + 1) * (kSelBins / C); i += kSelThreads)
      ca.ws.sel_hist[static_cast<size_t>(row) * kSelBins + i] = 0u;
  ECHO_TRACE_MARK(7);
  ECHO_TRACE_LAST(25);
}

}  // namespace echo

namespace echo_host {

int sm_count();

static int launch_topk_impl(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k,
                            int32_t *sel, float *kth, const echo::ClaimArgs &ca, int do_claim, cudaStream_t stream,
                            bool pdl) {
  const int rows = B * n_q;
  if (rows == 0) return ECHO_OK;
  const size_t fixed = sizeof(echo::SelSmem) + sizeof(echo::TopkExtra);
  // CTAs per row (one CTA per SM): kTopkCluster while the rows' clusters take at most
  // half the SMs; else 4 (many 8-CTA clusters wait longer for 8 free SMs of one GPC as the
  // kernel before drains); else 2 when only that fits one wave.  A slice that would not
  // fit shared memory keeps the larger cluster.
  const int sms = sm_count();
  auto fits = [&](int c) {
    const int ch = (((L_max + c - 1) / c) + 3) & ~3;
    return ch <= echo::kMaxChunk && fixed + static_cast<size_t>(ch) * sizeof(uint32_t) <= echo::kTopkSmemMax;
  };
  int C = echo::kTopkCluster;
  if (rows * C > sms / 2 && fits(4)) C = 4;
  if (C == 4 && rows * C > sms && fits(2)) C = 2;
  int chunk = (L_max + C - 1) / C;
  chunk = (chunk + 3) & ~3;
  if (chunk > echo::kMaxChunk) {
    set_error("top-k: L_max %d exceeds the supported %d", L_max, C * echo::kMaxChunk);
    return ECHO_ENOTSUP;
  }
  size_t smem = fixed + static_cast<size_t>(chunk > 0 ? chunk : 4) * sizeof(uint32_t);
  if (smem > static_cast<size_t>(echo::kTopkSmemMax)) {
    set_error("top-k: L_max %d needs more shared memory than a CTA has", L_max);
    return ECHO_ENOTSUP;
  }
  // the host rows of the slice go to shared memory too when they fit
  int stage_r2h = 0;
  if (do_claim && smem + static_cast<size_t>(chunk) * sizeof(int32_t) <= static_cast<size_t>(echo::kTopkSmemMax)) {
    smem += static_cast<size_t>(chunk) * sizeof(int32_t);
    stage_r2h = 1;
  }
  static std::atomic<bool> attr[kMaxDevices];
  if (int r = smem_limit_once(attr, echo::topk_kernel, echo::kTopkSmemMax, "top-k smem attribute")) return r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * C);
  cfg.blockDim = dim3(echo::kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, echo::topk_kernel, scores, ctx_len, n_q, L_max, k, chunk, sel, kth, ca, do_claim,
                         stage_r2h);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ECHO_OK;
}

int launch_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                float *kth, cudaStream_t stream) {
  echo::ClaimArgs none{};
  return launch_topk_impl(scores, ctx_len, B, n_q, L_max, k, sel, kth, none, 0, stream, false);
}

echo::PoolView pool_view(const echo_pool *p);
echo::Workspace workspace_view(const echo_workspace *w);

// top-k of the decode step: also claims the selected entries for the recall, and
// is launched programmatically after the indexer
int launch_topk_claim(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                      float *kth, const echo_pool *pool, const echo_workspace *ws, const int32_t *req_to_host,
                      int32_t clock, const int32_t *clock_dev, int32_t *status, cudaStream_t stream) {
  echo::ClaimArgs ca{};
  ca.pool = pool_view(pool);
  ca.ws = workspace_view(ws);
  ca.req_to_host = req_to_host;
  ca.clock = clock;
  ca.clock_dev = clock_dev;
  ca.status = status;
  return launch_topk_impl(scores, ctx_len, B, n_q, L_max, k, sel, kth, ca, 1, stream, true);
}

}  // namespace echo_host
