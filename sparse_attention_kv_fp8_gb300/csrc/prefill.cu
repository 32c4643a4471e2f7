// prefill.cu -- indexer score of a prefill chunk with the fused inter-query prefetch.
//
// ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"), section 6.2: during prefill
// the indexer takes the chunk's queries block by block, so while block i+1 is scored
// the tokens block i selects can already be fetched.  The exact top-k would slow the
// kernel, so each query's top-k is approximated: its scores, shifted by the predicted
// k-th score, go into a 256-bin histogram keyed by the top 8 bits; the top bins whose
// total stays within k are fetched (the guaranteed recall completes the rest).
// Section 6.3 (prefill kernel): each SM owns query blocks and all their key blocks;
// the prefetch warps histogram each score block and, once the query block is done,
// fetch the tokens above the threshold while the TMA and tensor-core warps already
// work on the next query block.
//
// sm_103a design (one persistent CTA per SM, 16 warps, so 128 registers a thread and
// no spills; query blocks of 4 tokens, so one tcgen05.mma of M = 128 keys x N = 256 =
// 4 queries x 64 heads x K = 32):
//   warp 0      TMA: the block's q (256 x 128 e4m3, two buffers) and its causal
//               range of 128-token k^I tiles into a 6-stage ring.
//   warp 1      tensor-core issuer: 4 MMAs per tile into one of two TMEM
//               accumulators of 256 columns.
//   warps 2-9   epilogue, two warpgroups on alternate tiles: ReLU, weight and head
//               sum per (token, query) in fp32, causal mask, score store, and the
//               block's histograms of shifted scores (shared memory, two buffers).
//   warps 10-15 prefetch: per finished block, the threshold bin of each query, then
//               a scan of the block's scores (just written, in L2) for the tokens
//               above it, residency test, tickets and host-row copies
//               (prefetch_rows.cuh), while the next block is being scored.
#include "echo_common.cuh"
#include "prefetch_rows.cuh"

namespace echo {

constexpr int kPQB = 4;                        // queries per block
constexpr int kPN = kHeads * kPQB;             // MMA N
constexpr int kPTile = 128;                    // keys per tile (MMA M)
constexpr int kPTileBytes = kPTile * kDim;     // 16 KB
constexpr int kPStages = 6;
constexpr int kPAcc = 2;                       // TMEM accumulators of kPN columns
constexpr int kPEpiGroups = 2;
constexpr int kPEpiWarps = 4 * kPEpiGroups;
constexpr int kPPfWarps = 6;                  // 16 warps in all: 128 registers a thread
constexpr int kPThreads = 32 * (2 + kPEpiWarps + kPPfWarps);
constexpr uint32_t kPQBytes = kPN * kDim;      // 32 KB
constexpr int kBins = 256;
constexpr int kPfBarrier = 1;                  // named barrier of the prefetch warps

struct PrefillParams {
  const float *w;          // [B][C][64]
  const int32_t *ctx_len;  // [B], the context including the chunk
  float *scores;           // [B][C][L_max]
  int32_t B, C, L_max, nb, n_units;
  // approximate top-k and prefetch (s_shift != nullptr)
  const float *s_shift;  // [B] predicted k-th score
  int32_t k;
  int32_t *thr_bin;   // [B][C] or nullptr
  int32_t *subset_n;  // [B][C] or nullptr
  // prefetch destinations (the field names prefetch_copy_batch reads)
  const int32_t *req_to_host;
  int32_t *host_to_gpu;
  int32_t n_h;
  const uint16_t *host_kv;
  uint16_t *stage_rows;
  int32_t *stage_host;
  int32_t *stage_count;
  int32_t stage_stride;
  int32_t cap_div;
  const int32_t *reserve;
  int32_t *reserve_ctl;
  int32_t *to_host;
  int32_t *prio;
  uint16_t *gpu_kv;
  int32_t n_g;
  int32_t *status;
};

struct alignas(16) PrefillCtl {
  uint64_t full[kPStages];
  uint64_t empty[kPStages];
  uint64_t tmem_full[kPAcc];
  uint64_t tmem_empty[kPAcc];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t hist_full[2];
  uint64_t hist_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int pf_ok;
  int thr[kPQB];
  float4 wsm[kPEpiWarps][kPN / 4];  // the block's head weights, per epilogue warp
};

// one query block of one request
struct Unit {
  int b, i0, nq;      // request, first query, queries in the block (<= kPQB)
  int valid[kPQB];    // keys query i0 + j sees (0 past nq)
  int lmax, tiles;    // keys of the block's last query, and its tiles
};

__device__ __forceinline__ Unit unit_of(const PrefillParams &P, int u) {
  Unit x;
  x.b = u / P.nb;
  x.i0 = (u % P.nb) * kPQB;
  x.nq = min(kPQB, P.C - x.i0);
  int32_t L = __ldg(P.ctx_len + x.b);
  if (L < 0 || L > P.L_max) {
    set_status(P.status, ECHO_DEV_BAD_INDEX);
    L = L < 0 ? 0 : P.L_max;
  }
#pragma unroll
  for (int j = 0; j < kPQB; ++j) x.valid[j] = j < x.nq ? query_valid_len(L, P.C, x.i0 + j) : 0;
  x.lmax = x.valid[x.nq - 1];
  x.tiles = (x.lmax + kPTile - 1) / kPTile;
  return x;
}

__device__ __forceinline__ void pmbar_drain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ void pf_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kPfBarrier), "n"(kPPfWarps * 32)); }

__global__ void __launch_bounds__(kPThreads, 1)
    prefill_indexer_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                           const PrefillParams P) {
  constexpr uint32_t kTmemCols = kPAcc * kPN;  // 512
  constexpr uint32_t kIdesc = idesc_e4m3_f32(kPTile, kPN);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *k_smem = smem;                                        // kPStages x 16 KB
  uint8_t *q_smem = smem + kPStages * kPTileBytes;               // 2 x 32 KB
  uint32_t *hist = reinterpret_cast<uint32_t *>(q_smem + 2 * kPQBytes);  // [2][kPQB][256]
  PrefillCtl *ctl = reinterpret_cast<PrefillCtl *>(hist + 2 * kPQB * kBins);
  volatile int *abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool approx = P.s_shift != nullptr;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int i = 0; i < kPAcc; ++i) {
      mbar_init(&ctl->tmem_full[i], 1);
      mbar_init(&ctl->tmem_empty[i], 4);  // the four warps of the group that reads it
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->hist_full[i], kPEpiWarps);
      mbar_init(&ctl->hist_empty[i], 1);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 2 * kPQB * kBins; i += kPThreads) hist[i] = 0;
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (elect_one()) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_q);
      const uint64_t policy = l2_policy_evict_last();  // every block of a request reads its keys
      int i = 0, qc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.n_units && ok; u += G) {
        const Unit x = unit_of(P, u);
        if (x.tiles == 0) continue;
        const int qb = qc & 1;
        if (qc >= 2 && !mbar_wait(&ctl->q_empty[qb], ((qc >> 1) - 1) & 1, abort, P.status)) break;
        mbar_arrive_expect_tx(&ctl->q_full[qb], kPQBytes);
        tma_load_2d(q_smem + qb * kPQBytes, &tmap_q, &ctl->q_full[qb], 0, (x.b * P.C + x.i0) * kHeads);
        ++qc;
        for (int t = 0; t < x.tiles; ++t, ++i) {
          const int s = i % kPStages;
          if (i >= kPStages && !mbar_wait(&ctl->empty[s], ((i / kPStages) & 1) ^ 1, abort, P.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->full[s], kPTileBytes);
          tma_load_3d_hint(k_smem + s * kPTileBytes, &tmap_k, &ctl->full[s], 0, t * kPTile, x.b, policy);
        }
      }
      if (*abort) {  // let every copy this thread started land before the CTA exits
        for (int j = i - kPStages < 0 ? 0 : i - kPStages; j < i; ++j)
          pmbar_drain(&ctl->full[j % kPStages], (j / kPStages) & 1);
        for (int c = qc - 2 < 0 ? 0 : qc - 2; c < qc; ++c) pmbar_drain(&ctl->q_full[c & 1], (c >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ===================== tensor-core issuer =====================
    if (elect_one()) {
      int i = 0, qc = 0, qb = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < P.n_units && ok; u += G) {
        const Unit x = unit_of(P, u);
        if (x.tiles == 0) continue;
        if (qc > 0) mma_commit(&ctl->q_empty[qb]);  // the previous block's q is no longer read
        qb = qc & 1;
        if (!mbar_wait(&ctl->q_full[qb], (qc >> 1) & 1, abort, P.status)) break;
        ++qc;
        for (int t = 0; t < x.tiles; ++t, ++i) {
          const int s = i % kPStages;
          const int ab = i % kPAcc;
          if (!mbar_wait(&ctl->full[s], (i / kPStages) & 1, abort, P.status) ||
              (i >= kPAcc && !mbar_wait(&ctl->tmem_empty[ab], ((i / kPAcc) & 1) ^ 1, abort, P.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(k_smem + s * kPTileBytes);
          const uint32_t b_addr = smem_u32(q_smem + qb * kPQBytes);
#pragma unroll
          for (int kk = 0; kk < kDim / 32; ++kk)
            mma_f8f6f4(tmem_base + ab * kPN, kmajor_sw128_desc(a_addr + kk * 32),
                       kmajor_sw128_desc(b_addr + kk * 32), kIdesc, kk > 0);
          mma_commit(&ctl->empty[s]);
          mma_commit(&ctl->tmem_full[ab]);
        }
      }
      mma_commit(&ctl->drain);  // every MMA issued above completes before TMEM is freed
      pmbar_drain(&ctl->drain, 0);
    }
  } else if (warp < 2 + kPEpiWarps) {
    // ===================== epilogue =====================
    const int e = warp - 2;
    const int grp = e / 4;
    const int quad = warp & 3;  // TMEM lanes this warp may read
    const int row = quad * 32 + lane;
    float4 *wsm4 = ctl->wsm[e];
    int i = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < P.n_units && ok; u += G, ++ui) {
      const Unit x = unit_of(P, u);
      const int hb = ui & 1;
      uint32_t *h = hist + hb * kPQB * kBins;
      if (approx && ui >= 2 && !mbar_wait(&ctl->hist_empty[hb], ((ui >> 1) - 1) & 1, abort, P.status)) break;
      const float shift = approx ? __ldg(P.s_shift + x.b) : 0.f;
      __syncwarp();
      for (int c = lane; c < kPN / 4; c += 32) {
        const int j = c / (kHeads / 4);
        wsm4[c] = j < x.nq ? __ldg(reinterpret_cast<const float4 *>(P.w + static_cast<size_t>(x.b * P.C + x.i0) *
                                                                               kHeads) + c)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncwarp();
      for (int t = 0; t < x.tiles; ++t, ++i) {
        if ((i & 1) != grp) continue;
        const int ab = i % kPAcc;
        if (!mbar_wait(&ctl->tmem_full[ab], (i / kPAcc) & 1, abort, P.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + ab * kPN;
        float sc[kPQB];
#pragma unroll
        for (int j = 0; j < kPQB; ++j) {
          sc[j] = 0.f;
          if (j >= x.nq) continue;  // warp-uniform
          float v0[32], v1[32];
          tmem_ld_32x32b_x32(taddr + j * kHeads, v0);
          tmem_ld_32x32b_x32(taddr + j * kHeads + 32, v1);
          tmem_wait_ld();
          reg_fence_32(v0);
          reg_fence_32(v1);
          const float4 *w4 = wsm4 + j * (kHeads / 4);
          float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);  // partial sums (0, 1), (2, 3)
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 wa = w4[h4], wb = w4[8 + h4];
            s01 = fma_relu2(wa.x, wa.y, v0[4 * h4 + 0], v0[4 * h4 + 1], s01);
            s23 = fma_relu2(wa.z, wa.w, v0[4 * h4 + 2], v0[4 * h4 + 3], s23);
            s01 = fma_relu2(wb.x, wb.y, v1[4 * h4 + 0], v1[4 * h4 + 1], s01);
            s23 = fma_relu2(wb.z, wb.w, v1[4 * h4 + 2], v1[4 * h4 + 3], s23);
          }
          sc[j] = (s01.x + s01.y) + (s23.x + s23.y);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->tmem_empty[ab]);
        const int p = t * kPTile + row;
#pragma unroll
        for (int j = 0; j < kPQB; ++j) {
          if (j >= x.nq) continue;
          const bool v = p < x.valid[j];
          if (v) P.scores[(static_cast<size_t>(x.b) * P.C + x.i0 + j) * P.L_max + p] = sc[j];
          if (approx) {
            // bin of the shifted score; lanes of one bin add together
            const uint32_t bin = v ? (score_key(sc[j] - shift) >> 24) : 0xFFFFFFFFu;
            const uint32_t same = __match_any_sync(0xffffffffu, bin);
            if (v && lane == __ffs(same) - 1) atomicAdd(h + j * kBins + bin, static_cast<uint32_t>(__popc(same)));
          }
        }
      }
      if (!ok) break;
      if (approx) {  // this warp's part of the block is in the histogram and the scores
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->hist_full[hb]);
      }
    }
  } else if (approx) {
    // ===================== approximate top-k and prefetch =====================
    const int pf = warp - 2 - kPEpiWarps;
    const int tid = pf * 32 + lane;
    const bool fetch = P.req_to_host != nullptr;  // a destination was given (else thresholds only)
    const bool direct = P.reserve != nullptr;
    const int32_t res_len = direct ? __ldg(P.reserve_ctl + 1) : 0;
    bool res_full = false;
    int ui = 0;
    for (int u = blockIdx.x; u < P.n_units; u += G, ++ui) {
      const Unit x = unit_of(P, u);
      const int hb = ui & 1;
      uint32_t *h = hist + hb * kPQB * kBins;
      if (tid == 0) ctl->pf_ok = mbar_wait(&ctl->hist_full[hb], (ui >> 1) & 1, abort, P.status) ? 1 : 0;
      pf_sync();
      if (!ctl->pf_ok) break;  // every prefetch warp leaves together
      // threshold bin of query j (warp j): lane l holds bins 255 - 8l .. 248 - 8l
      if (pf < x.nq) {
        uint32_t c[8], tot = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          c[r] = h[pf * kBins + 255 - 8 * lane - r];
          tot += c[r];
        }
        uint32_t inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const uint32_t all = __shfl_sync(0xffffffffu, inc, 31);
        const uint32_t kk = static_cast<uint32_t>(P.k);
        uint32_t run = inc - tot;  // scores in the bins above this lane's
        int thr = -2;
        uint32_t sub = 0;
        if (run <= kk) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (thr == -2 && run + c[r] > kk) {
              thr = 255 - 8 * lane - r;
              sub = run;
            }
            run += c[r];
          }
        }
        const uint32_t found = __ballot_sync(0xffffffffu, thr != -2);
        int t_bin = -1;
        uint32_t t_sub = all;  // every bin fits: all of them are taken
        if (found) {
          const int l = __ffs(found) - 1;
          t_bin = __shfl_sync(0xffffffffu, thr, l);
          t_sub = __shfl_sync(0xffffffffu, sub, l);
        }
        if (lane == 0) {
          ctl->thr[pf] = t_bin;
          const size_t q = static_cast<size_t>(x.b) * P.C + x.i0 + pf;
          if (P.thr_bin) P.thr_bin[q] = t_bin;
          if (P.subset_n) P.subset_n[q] = static_cast<int32_t>(t_sub);
        }
      }
      pf_sync();
      // the histogram buffer is free for the block after next
      for (int r = tid; r < kPQB * kBins; r += kPPfWarps * 32) h[r] = 0;
      pf_sync();
      if (tid == 0) mbar_arrive(&ctl->hist_empty[hb]);
      if (!fetch) continue;
      int thr[kPQB];
#pragma unroll
      for (int j = 0; j < kPQB; ++j) thr[j] = j < x.nq ? ctl->thr[j] : 256;
      const float shift = __ldg(P.s_shift + x.b);
      // tokens some query of the block puts above its threshold bin; the scores were
      // stored by this CTA's epilogue before its hist_full arrivals
      for (int p0 = 0; p0 < x.lmax; p0 += kPPfWarps * 32) {
        const int p = p0 + tid;
        bool cand = false;
        int32_t hrow = -1;
        if (p < x.lmax) {
#pragma unroll
          for (int j = 0; j < kPQB; ++j) {
            if (p < x.valid[j]) {
              const float s = __ldcg(P.scores + (static_cast<size_t>(x.b) * P.C + x.i0 + j) * P.L_max + p);
              cand |= static_cast<int>(score_key(s - shift) >> 24) > thr[j];
            }
          }
          if (cand) {
            hrow = __ldg(P.req_to_host + static_cast<size_t>(x.b) * P.L_max + p);
            if (hrow >= 0 && hrow < P.n_h) {
              cand = P.host_to_gpu[hrow] == kInf;
            } else {
              set_status(P.status, ECHO_DEV_BAD_INDEX);
              cand = false;
            }
          }
        }
        if (__any_sync(0xffffffffu, cand)) prefetch_copy_batch(P, cand, hrow, x.b, res_len, res_full);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace echo

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
namespace echo_host {

int sm_count();

typedef CUresult (*PFN_encodeTiledP)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);

static PFN_encodeTiledP encode_fn_p() {
  static PFN_encodeTiledP fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiledP>(p);
  }
  return fn;
}

static size_t prefill_smem_bytes() {
  return 1024 + echo::kPStages * echo::kPTileBytes + 2 * echo::kPQBytes +
         2 * echo::kPQB * echo::kBins * sizeof(uint32_t) + sizeof(echo::PrefillCtl);
}

int launch_prefill_indexer(const echo_prefill_args *a, cudaStream_t stream) {
  PFN_encodeTiledP enc = encode_fn_p();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled unavailable from the driver");
    return ECHO_ECUDA;
  }
  CUtensorMap tk, tq;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(echo::kDim), static_cast<cuuint64_t>(a->L_max),
                          static_cast<cuuint64_t>(a->B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(echo::kDim), static_cast<cuuint64_t>(a->L_max) * echo::kDim};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(echo::kDim), static_cast<cuuint32_t>(echo::kPTile), 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(a->k_index), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("tensor map for k_index failed (CUresult %d)", static_cast<int>(r));
      return ECHO_ECUDA;
    }
  }
  {
    // q rows: B * C * 64 of 128 bytes; a block reads 4 queries x 64 heads (rows past
    // the end read as zero, and rows of the next request are never used)
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(echo::kDim),
                          static_cast<cuuint64_t>(a->B) * a->C * echo::kHeads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(echo::kDim)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(echo::kDim), static_cast<cuuint32_t>(echo::kPN)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = enc(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a->q), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      set_error("tensor map for q failed (CUresult %d)", static_cast<int>(r));
      return ECHO_ECUDA;
    }
  }
  echo::PrefillParams P{};
  P.w = a->w;
  P.ctx_len = a->ctx_len;
  P.scores = a->scores;
  P.B = a->B;
  P.C = a->C;
  P.L_max = a->L_max;
  P.nb = (a->C + echo::kPQB - 1) / echo::kPQB;
  P.n_units = a->B * P.nb;
  P.status = a->dev_status;
  if (a->s_shift) {
    P.s_shift = a->s_shift;
    P.k = a->k;
    P.thr_bin = a->thr_bin;
    P.subset_n = a->subset_n;
    if (a->stage) {
      P.req_to_host = a->req_to_host;
      P.host_to_gpu = a->pool->host_token_to_gpu;
      P.n_h = a->pool->n_h;
      P.host_kv = a->pool->host_kv;
      if (a->stage->reserve) {
        P.reserve = a->stage->reserve;
        P.reserve_ctl = a->stage->reserve_ctl;
        P.to_host = a->pool->gpu_token_to_host;
        P.prio = a->pool->gpu_token_priority;
        P.gpu_kv = a->pool->gpu_kv;
        P.n_g = a->pool->n_g;
      } else {
        P.stage_rows = a->stage->rows;
        P.stage_host = a->stage->host_row;
        P.stage_count = a->stage->count;
        P.stage_stride = a->stage->stride;
        P.cap_div = a->stage->cap_div;
      }
    }
  }
  if (P.n_units == 0) return ECHO_OK;
  const int grid = P.n_units < sm_count() ? P.n_units : sm_count();
  const size_t smem = prefill_smem_bytes();
  static std::atomic<bool> attr[kMaxDevices];
  if (int r = smem_limit_once(attr, echo::prefill_indexer_kernel, static_cast<int>(smem), "prefill smem attribute"))
    return r;
  echo::prefill_indexer_kernel<<<grid, echo::kPThreads, smem, stream>>>(tk, tq, P);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "prefill indexer launch");
}

}  // namespace echo_host
