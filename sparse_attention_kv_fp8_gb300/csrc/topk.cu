// topk.cu -- exact top-k of the index scores (ECHO review, marsggbo.github.io,
// "OSDI'26 | ECHO", section 2: the indexer scores every cached token and the k
// highest (k = 2048 in DeepSeek-V3.2) go to the sparse MLA; section 6.2 names
// radix select over the score bits as the selection machinery).
//
// sm_103a design: one thread-block cluster of kTopkCluster CTAs per (request,
// query) row.  Each CTA keeps its slice of the row in shared memory as
// order-preserving uint32 keys (one global read).  Radix passes over the bits in
// which the row's keys differ (12-bit digits of key - min) find the k-th largest
// key exactly: each CTA histograms its slice, the cluster sums the histograms
// through distributed shared memory, and every CTA picks the same digit.  A final
// pass writes the selected indices in ascending order: per-thread segment counts,
// a block scan and a cluster scan give every selected token its output position
// (ties at the k-th value go to the lower index).
#include "cache_common.cuh"
#include "cluster_select.cuh"

ECHO_TRACE_UNIT(topk)

namespace echo {

constexpr int kTopkCluster = 8;
constexpr int kMaxChunk = 44 * 1024;  // keys per CTA kept in shared memory
constexpr int kCand = 1024;          // threshold-bin keys resolved by one CTA

struct alignas(16) TopkExtra {
  uint32_t cand_key[kCand];   // rank 0: keys of the threshold bin, from every CTA
  uint32_t cand_src[kCand];   // rank 0: the CTA each candidate came from
  uint32_t cand_n;            // rank 0: candidates received
  uint32_t above[kMaxCluster];  // rank 0: per-CTA count of keys in bins above the threshold bin
  uint32_t gc[kMaxCluster], ec[kMaxCluster];  // rank 0: per-CTA counts above / equal to T
  uint32_t T, needT, pg, pe;  // written by rank 0 into every CTA: threshold and this CTA's offsets
};

__global__ void __launch_bounds__(kSelThreads, 1)
    topk_kernel(const float *__restrict__ scores, const int32_t *__restrict__ ctx_len, int n_q, int L_max, int k,
                int chunk, int32_t *__restrict__ sel, float *__restrict__ kth, const ClaimArgs ca, int do_claim) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int row = blockIdx.x / C;
  const int b = row / n_q, j = row % n_q;
  const int lane = threadIdx.x & 31;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem *S = reinterpret_cast<SelSmem *>(smem_raw);
  TopkExtra *X = reinterpret_cast<TopkExtra *>(smem_raw + sizeof(SelSmem));
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem) + sizeof(TopkExtra));

  ECHO_TRACE_MARK(0);
  int L = __ldg(ctx_len + b);
  L = L < 0 ? 0 : (L > L_max ? L_max : L);
  const int Lr = query_valid_len(L, n_q, j);
  const int target = Lr < k ? Lr : k;
  const float *srow = scores + static_cast<size_t>(row) * L_max;
  int32_t *out = sel + static_cast<size_t>(row) * k;

  const int lo = rank * chunk;
  const int hi = lo + chunk < Lr ? lo + chunk : Lr;
  const int n_local = hi > lo ? hi - lo : 0;

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
  // the cluster-wide histogram is summed into every CTA's `tot`: clear it first
  for (int i = threadIdx.x; i < kMaxBins; i += kSelThreads) S->tot[i] = 0;
  if (threadIdx.x == 0) X->cand_n = 0;
  __syncthreads();
  ECHO_TRACE_MARK(1);

  // ---- the target-th largest key T, how many keys equal to T are taken (needT), and
  // this CTA's output offsets (keys above T and equal to T in lower CTAs)
  uint32_t T = 0, needT = 0, pg = 0, pe = 0;
  bool offsets_known = false;
  if (target > 0) {
    uint32_t kmin, kmax;
    sel_cluster_minmax(cl, S, mn, mx, kmin, kmax);  // also orders the clearing above before remote adds
    ECHO_TRACE_MARK(2);
    const uint32_t range = kmax - kmin;
    const int hb = range == 0 ? 0 : 32 - __clz(range);
    const int width = hb < kDigitBits ? hb : kDigitBits;
    const int shift = hb - width;
    const int nb = 1 << width;
    // first digit: local histogram, added into every CTA's total
    sel_histogram(S, n_local, 32, shift, nb, 0u, [&](int i, uint32_t &x) {
      x = keys[i] - kmin;
      return true;
    });
    for (int i = threadIdx.x; i < nb; i += kSelThreads) {
      const uint32_t v = S->hist[i];
      if (v)
        for (int r = 0; r < C; ++r) atomicAdd(cl.map_shared_rank(&S->tot[i], r), v);
    }
    cl.sync();
    ECHO_TRACE_MARK(3);
    // digit d holding the target-th largest key (descending running count)
    const int per = (nb + kSelThreads - 1) / kSelThreads;
    const int p0 = threadIdx.x * per;
    uint32_t cnt = 0, mine_above = 0;
    for (int u = 0; u < per; ++u)
      if (p0 + u < nb) cnt += S->tot[nb - 1 - (p0 + u)];
    uint32_t ex, dz, tt, tz;
    sel_block_scan2(cnt, 0, ex, dz, tt, tz, S);
    uint32_t run = ex;
    for (int u = 0; u < per; ++u) {
      const int idx = p0 + u;
      if (idx >= nb) break;
      const int bin = nb - 1 - idx;
      const uint32_t cb = S->tot[bin];
      if (run < static_cast<uint32_t>(target) && run + cb >= static_cast<uint32_t>(target)) {
        S->result[0] = static_cast<uint32_t>(bin);
        S->result[1] = run;
      }
      run += cb;
    }
    __syncthreads();
    const uint32_t d = S->result[0];
    const uint32_t need_d = static_cast<uint32_t>(target) - S->result[1];
    const uint32_t cnt_d = S->tot[d];
    // this CTA's keys in bins above d, and in bin d
    for (int i = threadIdx.x; i < nb; i += kSelThreads)
      if (static_cast<uint32_t>(i) > d) mine_above += S->hist[i];
    uint32_t in_d = S->hist[d];
    uint32_t ea, eb0, ta, tb0;
    sel_block_scan2(mine_above, 0, ea, eb0, ta, tb0, S);
    mine_above = ta;
    if (shift == 0) {
      // one key value per bin: T is exact, the local histogram gives the counts
      T = kmin + d;
      needT = need_d;
      sel_cluster_prefix2(cl, S, mine_above, in_d, pg, pe, tt, tz);
      offsets_known = true;
    } else if (cnt_d <= static_cast<uint32_t>(kCand)) {
      // ship the bin's keys to rank 0, which resolves T and every CTA's offsets
      TopkExtra *X0 = cl.map_shared_rank(X, 0);
      for (int base = (threadIdx.x & ~31); base < n_local; base += kSelThreads) {
        const int i = base + lane;
        const uint32_t key = i < n_local ? keys[i] : 0u;
        const bool cand = i < n_local && ((key - kmin) >> shift) == d;
        const uint32_t m = __ballot_sync(0xffffffffu, cand);
        if (!m) continue;
        uint32_t slot = 0;
        if (lane == __ffs(m) - 1) slot = atomicAdd(&X0->cand_n, static_cast<uint32_t>(__popc(m)));
        slot = __shfl_sync(0xffffffffu, slot, __ffs(m) - 1);
        if (cand) {
          const uint32_t at = slot + __popc(m & ((1u << lane) - 1));
          X0->cand_key[at] = key;
          X0->cand_src[at] = static_cast<uint32_t>(rank);
        }
      }
      if (threadIdx.x == 0) X0->above[rank] = mine_above;
      cl.sync();
      ECHO_TRACE_MARK(4);
      if (rank == 0) {
        const int nc = static_cast<int>(X->cand_n);
        if (threadIdx.x < kMaxCluster) {
          X->gc[threadIdx.x] = 0;
          X->ec[threadIdx.x] = 0;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nc; i += kSelThreads) {
          const uint32_t ki = X->cand_key[i];
          uint32_t greater = 0, equal = 0;
          for (int jj = 0; jj < nc; ++jj) {
            const uint32_t kj = X->cand_key[jj];
            greater += kj > ki;
            equal += kj == ki;
          }
          if (greater < need_d && need_d <= greater + equal) {
            S->result[0] = ki;
            S->result[1] = need_d - greater;
          }
        }
        __syncthreads();
        const uint32_t Tk = S->result[0];
        for (int i = threadIdx.x; i < nc; i += kSelThreads) {
          const uint32_t ki = X->cand_key[i];
          if (ki > Tk) atomicAdd(&X->gc[X->cand_src[i]], 1u);
          if (ki == Tk) atomicAdd(&X->ec[X->cand_src[i]], 1u);
        }
        __syncthreads();
        if (threadIdx.x < C) {
          uint32_t g0 = 0, e0 = 0;
          for (int r = 0; r < static_cast<int>(threadIdx.x); ++r) {
            g0 += X->above[r] + X->gc[r];
            e0 += X->ec[r];
          }
          TopkExtra *Xr = cl.map_shared_rank(X, static_cast<int>(threadIdx.x));
          Xr->T = Tk;
          Xr->needT = S->result[1];
          Xr->pg = g0;
          Xr->pe = e0;
        }
      }
      cl.sync();
      T = X->T;
      needT = X->needT;
      pg = X->pg;
      pe = X->pe;
      offsets_known = true;
    } else {
      // many keys share the threshold bin (ties or a clustered row): exact radix passes
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
  // equal keys; per-thread segments (odd length: conflict-free shared-memory reads)
  int seg = (n_local + kSelThreads - 1) / kSelThreads;
  seg |= 1;
  const int s0 = threadIdx.x * seg < n_local ? threadIdx.x * seg : n_local;
  const int s1 = s0 + seg < n_local ? s0 + seg : n_local;
  uint32_t g = 0, e = 0;
  if (target > 0)
    for (int i = s0; i < s1; ++i) {
      const uint32_t key = keys[i];
      g += key > T;
      e += key == T;
    }
  uint32_t eg, ee, tg, te;
  sel_block_scan2(g, e, eg, ee, tg, te, S);
  if (target > 0 && !offsets_known) {
    uint32_t gg, ge;
    sel_cluster_prefix2(cl, S, tg, te, pg, pe, gg, ge);
  }
  ECHO_TRACE_MARK(6);
  // the recall's claim of every selected entry (decode step): see cache_common.cuh
  const int32_t clock = do_claim ? (ca.clock_dev ? *ca.clock_dev : ca.clock) : 0;
  const int32_t *r2h = do_claim ? ca.req_to_host + static_cast<size_t>(b) * L_max : nullptr;
  const int f_row = row * k;
  if (target > 0) {
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
      if (pos < 0) continue;
      out[pos] = lo + i;
      if (do_claim) claim_entry(ca.pool, ca.ws, f_row + pos, __ldg(r2h + lo + i), clock, ca.status);
    }
  }
  for (int i = target + rank * kSelThreads + threadIdx.x; i < k; i += C * kSelThreads) {
    out[i] = -1;
    if (do_claim) ca.ws.entry_h[f_row + i] = -1;
  }
  if (rank == 0 && threadIdx.x == 0) kth[row] = target > 0 ? key_score(T) : -INFINITY;
  cl.sync();  // no CTA leaves while others may still read its shared memory
  ECHO_TRACE_MARK(7);
}

}  // namespace echo

namespace echo_host {

static int launch_topk_impl(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k,
                            int32_t *sel, float *kth, const echo::ClaimArgs &ca, int do_claim, cudaStream_t stream) {
  const int rows = B * n_q;
  if (rows == 0) return ECHO_OK;
  const int C = echo::kTopkCluster;
  int chunk = (L_max + C - 1) / C;
  chunk = (chunk + 3) & ~3;
  if (chunk > echo::kMaxChunk) {
    set_error("top-k: L_max %d exceeds the supported %d", L_max, C * echo::kMaxChunk);
    return ECHO_ENOTSUP;
  }
  const size_t smem = sizeof(echo::SelSmem) + sizeof(echo::TopkExtra) +
                      static_cast<size_t>(chunk > 0 ? chunk : 4) * sizeof(uint32_t);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(echo::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return cuda_fail(e, "top-k smem attribute");
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows * C);
  cfg.blockDim = dim3(echo::kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaError_t e =
      cudaLaunchKernelEx(&cfg, echo::topk_kernel, scores, ctx_len, n_q, L_max, k, chunk, sel, kth, ca, do_claim);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ECHO_OK;
}

int launch_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                float *kth, cudaStream_t stream) {
  echo::ClaimArgs none{};
  return launch_topk_impl(scores, ctx_len, B, n_q, L_max, k, sel, kth, none, 0, stream);
}

echo::PoolView pool_view(const echo_pool *p);
echo::Workspace workspace_view(const echo_workspace *w);

// top-k of the decode step: also claims the selected entries for the recall
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
  return launch_topk_impl(scores, ctx_len, B, n_q, L_max, k, sel, kth, ca, 1, stream);
}

}  // namespace echo_host
