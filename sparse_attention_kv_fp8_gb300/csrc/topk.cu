// topk.cu -- exact top-k of the index scores (ECHO review, marsggbo.github.io,
// "OSDI'26 | ECHO", section 2: the indexer scores every cached token and the k
// highest (k = 2048 in DeepSeek-V3.2) go to the sparse MLA; section 6.2 names
// radix select over the score bits as the selection machinery).
//
// sm_103a design: one thread-block cluster of kCluster CTAs per (request, query)
// row.  Each CTA keeps its slice of the row in shared memory as order-preserving
// uint32 keys (one global read).  Three radix passes (11, 11, 10 bits) find the
// k-th largest key exactly: each CTA histograms its slice, the cluster sums the
// histograms through distributed shared memory, and every CTA picks the same
// digit.  A final pass writes the selected indices in ascending order: per-thread
// segment counts, a block scan and a cluster scan give every selected token its
// output position (ties at the k-th value go to the lower index).
#include <cooperative_groups.h>

#include "echo_common.cuh"

namespace cg = cooperative_groups;

namespace echo {

constexpr int kCluster = 8;
constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kMaxBins = 2048;
constexpr int kMaxChunk = 49152;  // keys per CTA kept in shared memory (192 KB)

struct TopkSmem {
  uint32_t hist[kMaxBins];
  uint32_t tot[kMaxBins];
  uint32_t warp_a[kTopkWarps];
  uint32_t warp_b[kTopkWarps];
  uint32_t cta_g, cta_e;  // this CTA's count of keys above / equal to the k-th key
  uint32_t digit, above;
};

// inclusive scan of two counters over the block; returns exclusive prefixes
__device__ __forceinline__ void block_scan2(uint32_t a, uint32_t b, uint32_t &ea, uint32_t &eb,
                                            uint32_t &ta, uint32_t &tb, TopkSmem *S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
    }
  }
  if (lane == 31) {
    S->warp_a[warp] = ia;
    S->warp_b[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t wa = S->warp_a[lane], wb = S->warp_b[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t xa = __shfl_up_sync(0xffffffffu, wa, o), xb = __shfl_up_sync(0xffffffffu, wb, o);
      if (lane >= o) {
        wa += xa;
        wb += xb;
      }
    }
    S->warp_a[lane] = wa;
    S->warp_b[lane] = wb;
  }
  __syncthreads();
  const uint32_t pa = warp ? S->warp_a[warp - 1] : 0, pb = warp ? S->warp_b[warp - 1] : 0;
  ea = pa + ia - a;
  eb = pb + ib - b;
  ta = S->warp_a[kTopkWarps - 1];
  tb = S->warp_b[kTopkWarps - 1];
  __syncthreads();
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kTopkThreads, 1)
    topk_kernel(const float *__restrict__ scores, const int32_t *__restrict__ ctx_len, int n_q,
                int L_max, int k, int chunk, int32_t *__restrict__ sel, float *__restrict__ kth) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.x / kCluster;
  const int b = row / n_q, j = row % n_q;
  extern __shared__ uint8_t smem_raw[];
  TopkSmem *S = reinterpret_cast<TopkSmem *>(smem_raw);
  uint32_t *keys = reinterpret_cast<uint32_t *>(smem_raw + sizeof(TopkSmem));

  int L = __ldg(ctx_len + b);
  L = L < 0 ? 0 : (L > L_max ? L_max : L);
  const int Lr = query_valid_len(L, n_q, j);
  const int target = Lr < k ? Lr : k;
  const float *srow = scores + static_cast<size_t>(row) * L_max;
  int32_t *out = sel + static_cast<size_t>(row) * k;

  const int lo = rank * chunk;
  const int hi = lo + chunk < Lr ? lo + chunk : Lr;
  const int n_local = hi > lo ? hi - lo : 0;

  // ---- load the slice as keys (16-byte loads when the slice is aligned)
  if (((reinterpret_cast<uintptr_t>(srow + lo) & 15) == 0)) {
    const int nv = n_local >> 2;
    const float4 *src = reinterpret_cast<const float4 *>(srow + lo);
    for (int i = threadIdx.x; i < nv; i += kTopkThreads) {
      float4 v = __ldcg(src + i);
      keys[4 * i + 0] = score_key(v.x);
      keys[4 * i + 1] = score_key(v.y);
      keys[4 * i + 2] = score_key(v.z);
      keys[4 * i + 3] = score_key(v.w);
    }
    for (int i = (nv << 2) + threadIdx.x; i < n_local; i += kTopkThreads) keys[i] = score_key(__ldcg(srow + lo + i));
  } else {
    for (int i = threadIdx.x; i < n_local; i += kTopkThreads) keys[i] = score_key(__ldcg(srow + lo + i));
  }
  __syncthreads();

  // ---- three radix passes: find the target-th largest key T
  uint32_t prefix = 0, pmask = 0, need = static_cast<uint32_t>(target);
  if (target > 0) {
    const int shifts[3] = {21, 10, 0};
    const int bins_of[3] = {2048, 2048, 1024};
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = shifts[pass], nb = bins_of[pass];
      const uint32_t dmask = static_cast<uint32_t>(nb - 1);
      for (int i = threadIdx.x; i < nb; i += kTopkThreads) S->hist[i] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n_local; i += kTopkThreads) {
        const uint32_t key = keys[i];
        if ((key & pmask) == prefix) atomicAdd(&S->hist[(key >> shift) & dmask], 1u);
      }
      __syncthreads();
      cluster.sync();  // every slice histogram complete
      for (int i = threadIdx.x; i < nb; i += kTopkThreads) {
        uint32_t s = 0;
#pragma unroll
        for (int r = 0; r < kCluster; ++r) s += cluster.map_shared_rank(S->hist, r)[i];
        S->tot[i] = s;
      }
      __syncthreads();
      // suffix counts from the top digit down; thread t owns reversed bins 2t, 2t+1
      const int r0 = 2 * threadIdx.x, r1 = r0 + 1;
      const uint32_t c0 = r0 < nb ? S->tot[nb - 1 - r0] : 0;
      const uint32_t c1 = r1 < nb ? S->tot[nb - 1 - r1] : 0;
      uint32_t ex, dummy, tot, tot2;
      block_scan2(c0 + c1, 0, ex, dummy, tot, tot2, S);
      const uint32_t suf0 = ex + c0, suf1 = ex + c0 + c1;  // counts of bins >= digit
      if (r0 < nb && suf0 >= need && ex < need) {
        S->digit = static_cast<uint32_t>(nb - 1 - r0);
        S->above = ex;
      }
      if (r1 < nb && suf1 >= need && suf0 < need) {
        S->digit = static_cast<uint32_t>(nb - 1 - r1);
        S->above = suf0;
      }
      __syncthreads();
      prefix |= S->digit << shift;
      pmask |= dmask << shift;
      need -= S->above;
      cluster.sync();  // remote histogram reads done before the next pass clears them
    }
  }
  const uint32_t T = prefix;  // the target-th largest key; `need` keys equal to T are taken

  // ---- positions: selected iff key > T, or key == T among the first `need` equal keys
  const int seg = (n_local + kTopkThreads - 1) / kTopkThreads;
  const int s0 = threadIdx.x * seg;
  const int s1 = s0 + seg < n_local ? s0 + seg : n_local;
  uint32_t g = 0, e = 0;
  if (target > 0)
    for (int i = s0; i < s1; ++i) {
      const uint32_t key = keys[i];
      g += key > T;
      e += key == T;
    }
  uint32_t eg, ee, tg, te;
  block_scan2(g, e, eg, ee, tg, te, S);
  if (threadIdx.x == 0) {
    S->cta_g = tg;
    S->cta_e = te;
  }
  cluster.sync();
  uint32_t base_g = 0, base_e = 0;
  for (int r = 0; r < rank; ++r) {
    TopkSmem *R = cluster.map_shared_rank(S, r);
    base_g += R->cta_g;
    base_e += R->cta_e;
  }
  if (target > 0) {
    uint32_t gb = base_g + eg, eb = base_e + ee;
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
  for (int i = target + rank * kTopkThreads + threadIdx.x; i < k; i += kCluster * kTopkThreads) out[i] = -1;
  if (rank == 0 && threadIdx.x == 0) kth[row] = target > 0 ? key_score(T) : -INFINITY;
  cluster.sync();  // no CTA leaves while others may still read its shared memory
}

}  // namespace echo

namespace echo_host {

int launch_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                float *kth, cudaStream_t stream) {
  const int rows = B * n_q;
  if (rows == 0) return ECHO_OK;
  int chunk = (L_max + echo::kCluster - 1) / echo::kCluster;
  chunk = (chunk + 3) & ~3;
  if (chunk > echo::kMaxChunk) {
    set_error("top-k: L_max %d exceeds the supported %d", L_max, echo::kCluster * echo::kMaxChunk);
    return ECHO_ENOTSUP;
  }
  const size_t smem = sizeof(echo::TopkSmem) + static_cast<size_t>(chunk > 0 ? chunk : 4) * sizeof(uint32_t);
  static size_t smem_set = 0;
  if (smem > smem_set) {
    cudaError_t e = cudaFuncSetAttribute(echo::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem < 232448 ? 232448 : smem));
    if (e != cudaSuccess) return cuda_fail(e, "top-k smem attribute");
    smem_set = 232448;
  }
  echo::topk_kernel<<<rows * echo::kCluster, echo::kTopkThreads, smem, stream>>>(scores, ctx_len, n_q, L_max, k,
                                                                                  chunk, sel, kth);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ECHO_OK;
}

}  // namespace echo_host
