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
#include "cluster_select.cuh"

ECHO_TRACE_UNIT(topk)

namespace echo {

constexpr int kTopkCluster = 8;
constexpr int kMaxChunk = 48 * 1024;  // keys per CTA kept in shared memory

__global__ void __launch_bounds__(kSelThreads, 1)
    topk_kernel(const float *__restrict__ scores, const int32_t *__restrict__ ctx_len, int n_q, int L_max, int k,
                int chunk, int32_t *__restrict__ sel, float *__restrict__ kth) {
  cg::cluster_group cl = cg::this_cluster();
  const int C = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  const int row = blockIdx.x / C;
  const int b = row / n_q, j = row % n_q;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelSmem *S = reinterpret_cast<SelSmem *>(smem_raw);
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelSmem));  // SelSmem is 16-byte aligned in size

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
  __syncthreads();

  ECHO_TRACE_MARK(1);
  // ---- the target-th largest key T and how many keys equal to T are taken
  uint32_t T = 0, need = 0;
  if (target > 0) {
    uint32_t kmin, kmax;
    sel_cluster_minmax(cl, S, mn, mx, kmin, kmax);
    ECHO_TRACE_MARK(2);
    sel_radix_select(cl, S, n_local, kmin, kmax, static_cast<uint32_t>(target), true,
                     [&](int i, uint32_t &key) {
                       key = keys[i];
                       return true;
                     },
                     T, need);
  }

  ECHO_TRACE_MARK(3);
  // ---- ascending output: selected iff key > T, or key == T among the first `need`
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
  uint32_t pg, pe, gg, ge;
  sel_cluster_prefix2(cl, S, tg, te, pg, pe, gg, ge);
  ECHO_TRACE_MARK(4);
  if (target > 0) {
    uint32_t gb = pg + eg, eb = pe + ee;
    for (int i = s0; i < s1; ++i) {
      const uint32_t key = keys[i];
      if (key > T) {
        out[gb + (eb < need ? eb : need)] = lo + i;
        ++gb;
      } else if (key == T) {
        if (eb < need) out[gb + eb] = lo + i;
        ++eb;
      }
    }
  }
  for (int i = target + rank * kSelThreads + threadIdx.x; i < k; i += C * kSelThreads) out[i] = -1;
  if (rank == 0 && threadIdx.x == 0) kth[row] = target > 0 ? key_score(T) : -INFINITY;
  ECHO_TRACE_MARK(5);
  cl.sync();  // no CTA leaves while others may still read its shared memory
  ECHO_TRACE_MARK(6);
}

}  // namespace echo

namespace echo_host {

int launch_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                float *kth, cudaStream_t stream) {
  const int rows = B * n_q;
  if (rows == 0) return ECHO_OK;
  const int C = echo::kTopkCluster;
  int chunk = (L_max + C - 1) / C;
  chunk = (chunk + 3) & ~3;
  if (chunk > echo::kMaxChunk) {
    set_error("top-k: L_max %d exceeds the supported %d", L_max, C * echo::kMaxChunk);
    return ECHO_ENOTSUP;
  }
  const size_t smem = sizeof(echo::SelSmem) + static_cast<size_t>(chunk > 0 ? chunk : 4) * sizeof(uint32_t);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, echo::topk_kernel, scores, ctx_len, n_q, L_max, k, chunk, sel, kth);
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ECHO_OK;
}

}  // namespace echo_host
