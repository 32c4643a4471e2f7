// indexer.cu -- DSA lightning-indexer score with the fused lossless prefetch.
//
// ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"): section 2 "DSA indexer"
// gives s(t,s) = sum_h w_{h,t} ReLU(q_{h,t} . k_s) with H_index = 64, d_index = 128
// and FP8 q/k; section 6.3 describes the decode kernel as a warp-specialised
// pipeline (TMA warps load K blocks, GEMM warps write scores, prefetch warps
// compare scores with the predicted k-th score and load rows from host memory),
// one SM per query vector and a slice of the K cache.
//
// sm_103a design (one persistent CTA per SM, 14 warps for one query token, 16 for two;
// up to 128 registers a thread):
//   warp 0      TMA producer: 128-token K tiles (16 KB, 128B-swizzled) into a
//               10-stage shared-memory ring; the request's q (64*n_q x 128 e4m3)
//               into one of two q buffers; the tiles' host rows (req_to_host).
//   warp 1      tensor-core issuer: per tile, 4 x tcgen05.mma kind::f8f6f4
//               (M = 128 tokens, N = 64*n_q heads, K = 32) into one of four TMEM
//               accumulators, so the MMA runs ahead of the epilogue.
//   warps 2-9   epilogue (2-13 for two query tokens), two (three) warpgroups taking
//               tiles in turn: tcgen05.ld one token row per thread, ReLU, weight, sum
//               over heads in fp32, store the score; threshold test against the
//               predicted k-th score; candidates go to a per-warp queue.
//   warps 10-13 prefetch (14-15 for two query tokens), each serving two (six)
//               epilogue warps' queues: residency test and tickets for the queued
//               tokens, then copy their host rows (1152 B, 16-byte loads of the
//               pinned, mapped host pool) into the HBM staging area, or straight into
//               the GPU-pool slots the last recall set aside (direct to slot).
// The kernel is HBM-bound: 128 + 4*n_q bytes per token against 2*64*128*n_q
// FLOP, far below the FP8 ridge point.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "cache_common.cuh"
#include "prefetch_rows.cuh"

ECHO_TRACE_UNIT(indexer)

namespace echo {

constexpr int kTileTokens = 128;
constexpr int kTileBytes = kTileTokens * kDim;  // 16 KB
constexpr int kStages = 10;
// Warp roles per query count: epilogue warpgroups taking tiles in turn, and prefetch
// warps each serving kEpiWarps / kPfWarps queues.  Two query tokens double the epilogue's
// TMEM reads and sums per tile, so that kernel has a third epilogue warpgroup (the four
// TMEM accumulators cover three groups and the MMA) and two prefetch warps: 16 warps,
// 128 registers a thread.
template <int NQ>
struct Roles {
  static constexpr int kEpiGroups = NQ == 1 ? 2 : 3;
  static constexpr int kEpiWarps = 4 * kEpiGroups;
  static constexpr int kPfWarps = NQ == 1 ? 4 : 2;
  static constexpr int kThreads = 32 * (2 + kEpiWarps + kPfWarps);
  static_assert(kEpiWarps % kPfWarps == 0, "whole queues per prefetch warp");
};

constexpr int kAcc = 4;            // TMEM accumulators (MMA runs up to 3 tiles ahead of the epilogue)
constexpr int kQueueCap = 64;      // entries per epilogue -> prefetch queue
// prefetching while scoring: each epilogue warpgroup of a CTA with at least
// kPfTailMin tiles per group queues no candidate from its last kPfTailTiles tiles
// (their host reads would land after the CTA's scoring ends and only lengthen the
// kernel; the recall fetches such rows if they are selected).  Into the staging area
// the last four tiles are cut; direct to slot only the last two, since a row placed
// there spares the recall a whole copy, where a staged row still needs one.
constexpr int kPfTailTiles = 4;
constexpr int kPfTailTilesDirect = 2;
constexpr int kPfTailMin = 8;
// host rows of the tiles (req_to_host slices, 128 x int32) staged by TMA for the
// epilogue: a ring the producer may refill only after the epilogue read the tile
// kR tiles back, which the k^I ring and the TMEM accumulators already guarantee
constexpr int kR = kStages + kAcc;
constexpr int kRowMapBytes = kTileTokens * 4;

struct IndexerParams {
  const float *w;
  const int32_t *ctx_len;
  float *scores;
  int32_t B, L_max;
  // fused prefetch (enabled when s_hat != nullptr)
  const float *s_hat;
  const int32_t *req_to_host;
  int32_t *host_to_gpu;  // written only by the direct-to-slot prefetch
  int32_t n_h;
  const uint16_t *host_kv;
  uint16_t *stage_rows;
  int32_t *stage_host;
  int32_t *stage_count;
  int32_t stage_stride;
  int32_t cap_div;
  int32_t pf_while_scoring;  // drop candidates still queued once the CTA's scoring is done
  // direct-to-slot prefetch (reserve != nullptr): the reserved slots, the ticket
  // counter / reserve length, and the pool arrays a placed row updates
  const int32_t *reserve;
  int32_t *reserve_ctl;
  int32_t *to_host;
  int32_t *prio;
  uint16_t *gpu_kv;
  int32_t n_g;
  int32_t *status;
  int32_t r2h_tma;  // the tiles' host rows come by TMA (needs L_max % 4 == 0)
  // decode step: per score row (b * n_q + j < kSelHintRows) a histogram of the score
  // keys over the window sel_hint[row] (when valid), read by the top-k that follows
  uint32_t *sel_hist;
  const int4 *sel_hint;
};

template <int EW>  // epilogue warps
struct alignas(16) IndexerCtl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tmem_full[kAcc];
  uint64_t tmem_empty[kAcc];
  uint64_t q_full[2];
  uint64_t q_empty[2];
  uint64_t drain;
  uint64_t r2h_full[kR];
  uint32_t tmem_base;
  int abort;
  int first_b, first_t, n_tiles;
  int queue_tail[EW];
  int queue_head[EW];
  int queue_done[EW];
  int queue[EW][kQueueCap];    // token ids b * L_max + p that passed the threshold
  int queue_h[EW][kQueueCap];  // their host rows (when the tiles' host rows are staged)
  float4 wsm[EW][2 * kHeads / 4];  // head weights of the current request, per epilogue warp
  uint32_t hwin[EW][2][2];         // the current request's histogram windows {low key, shift}
};

__device__ __forceinline__ int tiles_of(int L) { return (L + kTileTokens - 1) / kTileTokens; }

// next (request, tile) in the flattened sequence of non-empty tiles
__device__ __forceinline__ void next_tile(const IndexerParams &P, int &b, int &t) {
  ++t;
  while (b < P.B && t >= tiles_of(clamp_ctx(__ldg(P.ctx_len + b), P.L_max))) {
    ++b;
    t = 0;
  }
}

// Bounded wait used while unwinding: ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitLimitNs) return;
}

template <int NQ>
__global__ void __launch_bounds__(Roles<NQ>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_r, const IndexerParams P) {
  constexpr int N = kHeads * NQ;               // MMA N: all heads of all queries
  constexpr int kEpiGroups = Roles<NQ>::kEpiGroups, kEpiWarps = Roles<NQ>::kEpiWarps;
  constexpr int kPfWarps = Roles<NQ>::kPfWarps;
  constexpr uint32_t kQBytes = N * kDim;       // q of one request
  constexpr uint32_t kTmemCols = kAcc * N;     // 256 (NQ = 1) or 512 (NQ = 2) columns
  constexpr uint32_t kIdesc = idesc_e4m3_f32(kTileTokens, N);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *k_smem = smem;                                  // kStages x 16 KB
  uint8_t *q_smem = smem + kStages * kTileBytes;           // 2 x kQBytes
  int32_t *r_smem = reinterpret_cast<int32_t *>(q_smem + 2 * kQBytes);  // kR x 128 host rows
  using Ctl = IndexerCtl<Roles<NQ>::kEpiWarps>;
  Ctl *ctl = reinterpret_cast<Ctl *>(q_smem + 2 * kQBytes + kR * kRowMapBytes);
  volatile int *abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool prefetch = P.s_hat != nullptr;
  pdl_launch_dependents();  // the top-k may be scheduled as SMs free up; it waits for completion
  ECHO_TRACE_FIRST(24);

  // ---- work split: the non-empty tiles of all requests, evenly over the grid.  Warp
  // 0 reads the context lengths 32 at a time (one round trip for up to 32 requests).
  if (warp == 0) {
    int total = 0;
    for (int b0 = 0; b0 < P.B; b0 += 32) {
      const int b = b0 + lane;
      int nt = 0;
      if (b < P.B) {
        const int32_t L = __ldg(P.ctx_len + b);
        if (L < 0 || L > P.L_max) set_status(P.status, ECHO_DEV_BAD_INDEX);
        nt = tiles_of(clamp_ctx(L, P.L_max));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) nt += __shfl_xor_sync(0xffffffffu, nt, o);
      total += nt;
    }
    const int v0 = static_cast<int>((static_cast<long long>(total) * blockIdx.x) / gridDim.x);
    const int v1 = static_cast<int>((static_cast<long long>(total) * (blockIdx.x + 1)) / gridDim.x);
    // the request holding tile v0: the first whose inclusive tile count passes v0
    int acc = 0, first_b = P.B, first_t = 0;
    for (int b0 = 0; b0 < P.B && first_b == P.B; b0 += 32) {
      const int b = b0 + lane;
      const int nt = b < P.B ? tiles_of(clamp_ctx(__ldg(P.ctx_len + b), P.L_max)) : 0;
      int inc = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
      }
      const uint32_t hit = __ballot_sync(0xffffffffu, b < P.B && v0 < acc + inc);
      if (hit) {
        const int l = __ffs(hit) - 1;
        first_b = b0 + l;
        first_t = v0 - (acc + __shfl_sync(0xffffffffu, inc - nt, l));
      }
      acc += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) {
      ctl->first_b = first_b;
      ctl->first_t = first_b < P.B ? first_t : 0;
      ctl->n_tiles = v1 - v0;
      ctl->abort = 0;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(&ctl->tmem_full[i], 1);
      mbar_init(&ctl->tmem_empty[i], 4);  // the four warps of the group that reads it
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
    }
    mbar_init(&ctl->drain, 1);
    for (int i = 0; i < kR; ++i) mbar_init(&ctl->r2h_full[i], 1);
    for (int e = 0; e < kEpiWarps; ++e) {
      ctl->queue_tail[e] = 0;
      ctl->queue_head[e] = 0;
      ctl->queue_done[e] = 0;
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  ECHO_TRACE_FIRST(28);
  ECHO_TRACE_LAST(29);

  const int n_tiles = ctl->n_tiles;
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // ===================== TMA producer =====================
    if (elect_one()) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_q);
      const bool rows_by_tma = prefetch && P.r2h_tma;
      if (rows_by_tma) tma_prefetch_desc(&tmap_r);
      const uint64_t policy = l2_policy_evict_first();
      int b = ctl->first_b, t = ctl->first_t, cur_b = -1, qcount = 0, issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        if (b != cur_b) {
          const int qb = qcount & 1;
          if (qcount >= 2 && !mbar_wait(&ctl->q_empty[qb], ((qcount >> 1) - 1) & 1, abort, P.status)) break;
          mbar_arrive_expect_tx(&ctl->q_full[qb], kQBytes);
          tma_load_2d(q_smem + qb * kQBytes, &tmap_q, &ctl->q_full[qb], 0, b * N);
          cur_b = b;
          ++qcount;
        }
        const int s = i % kStages;
        if (i >= kStages && !mbar_wait(&ctl->empty[s], ((i / kStages) & 1) ^ 1, abort, P.status)) break;
        mbar_arrive_expect_tx(&ctl->full[s], kTileBytes);
        tma_load_3d_hint(k_smem + s * kTileBytes, &tmap_k, &ctl->full[s], 0, t * kTileTokens, b, policy);
        if (rows_by_tma) {  // the tile's host rows, for the epilogue's prefetch candidates
          const int rs = i % kR;
          mbar_arrive_expect_tx(&ctl->r2h_full[rs], kRowMapBytes);
          tma_load_2d(r_smem + rs * kTileTokens, &tmap_r, &ctl->r2h_full[rs], t * kTileTokens, b);
        }
        ++issued;
        next_tile(P, b, t);
      }
      if (*abort) {
        // let every copy this thread started land before the CTA exits
        for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
          mbar_drain(&ctl->full[i % kStages], (i / kStages) & 1);
        for (int c = qcount - 2 < 0 ? 0 : qcount - 2; c < qcount; ++c) mbar_drain(&ctl->q_full[c & 1], (c >> 1) & 1);
        if (rows_by_tma)
          for (int i = issued - kR < 0 ? 0 : issued - kR; i < issued; ++i)
            mbar_drain(&ctl->r2h_full[i % kR], (i / kR) & 1);
      }
    }
  } else if (warp == 1) {
    // ===================== tensor-core issuer =====================
    if (elect_one()) {
      int b = ctl->first_b, t = ctl->first_t, cur_b = -1, qcount = 0, qb = 0;
      for (int i = 0; i < n_tiles; ++i) {
        if (b != cur_b) {
          if (cur_b >= 0) mma_commit(&ctl->q_empty[qb]);  // previous q no longer read
          qb = qcount & 1;
          if (!mbar_wait(&ctl->q_full[qb], (qcount >> 1) & 1, abort, P.status)) break;
          cur_b = b;
          ++qcount;
        }
        const int s = i % kStages;
        if (!mbar_wait(&ctl->full[s], (i / kStages) & 1, abort, P.status)) break;
        if (i == 0) ECHO_TRACE_LAST_HERE(30);
        const int ab = i % kAcc;
        if (i >= kAcc && !mbar_wait(&ctl->tmem_empty[ab], ((i / kAcc) & 1) ^ 1, abort, P.status)) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(k_smem + s * kTileBytes);
        const uint32_t b_addr = smem_u32(q_smem + qb * kQBytes);
#pragma unroll
        for (int kk = 0; kk < kDim / 32; ++kk)
          mma_f8f6f4(tmem_base + ab * N, kmajor_sw128_desc(a_addr + kk * 32),
                     kmajor_sw128_desc(b_addr + kk * 32), kIdesc, kk > 0);
        mma_commit(&ctl->empty[s]);
        mma_commit(&ctl->tmem_full[ab]);
        next_tile(P, b, t);
      }
      // every MMA issued above completes before the accumulators are freed
      mma_commit(&ctl->drain);
      mbar_drain(&ctl->drain, 0);
    }
  } else if (warp < 2 + kEpiWarps) {
    // ===================== epilogue =====================
    // group g takes tiles g, g + kEpiGroups, ... so two or three warps per SM sub-partition
    // hide each other's TMEM-load and FMA latency
    const int e = warp - 2;
    const int grp = e / 4;
    const int quad = warp & 3;  // TMEM lanes this warp may read
    const int row = quad * 32 + lane;
    float4 *wsm4 = ctl->wsm[e];
    int b = ctl->first_b, t = ctl->first_t, cur_b = -1;
    for (int u = 0; u < grp; ++u) next_tile(P, b, t);
    const bool pf_cut = P.pf_while_scoring && n_tiles >= kPfTailMin * kEpiGroups;
    const int pf_tail = (P.reserve != nullptr ? kPfTailTilesDirect : kPfTailTiles) * kEpiGroups;
    float shat[NQ];
    int valid[NQ];
    uint32_t hist_on = 0;  // bit j: query j's row has a selection histogram (window in hwin[e][j])
    int tail = 0;  // queue tail, kept by every lane (lane 0 publishes it)
    for (int i = grp; i < n_tiles; i += kEpiGroups) {
      if (b != cur_b) {
        __syncwarp();
        for (int x = lane; x < N / 4; x += 32)
          wsm4[x] = __ldg(reinterpret_cast<const float4 *>(P.w + static_cast<size_t>(b) * N) + x);
        __syncwarp();
        const int L = clamp_ctx(__ldg(P.ctx_len + b), P.L_max);
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          valid[j] = query_valid_len(L, NQ, j);
          shat[j] = prefetch ? __ldg(P.s_hat + b * NQ + j) : 0.f;
        }
        hist_on = 0;
        if (P.sel_hist && (b + 1) * NQ <= kSelHintRows) {
          __syncwarp();
          if (lane < NQ) {
            const int4 h = P.sel_hint[b * NQ + lane];
            ctl->hwin[e][lane][0] = static_cast<uint32_t>(h.x);
            ctl->hwin[e][lane][1] = static_cast<uint32_t>(h.y);
            hist_on = h.z ? 1u << lane : 0u;
          }
          __syncwarp();  // the windows are in shared memory before any lane reads them
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) hist_on |= __shfl_xor_sync(0xffffffffu, hist_on, o);
        }
        cur_b = b;
      }
      const int ab = i % kAcc;
      if (!mbar_wait(&ctl->tmem_full[ab], (i / kAcc) & 1, abort, P.status)) break;
      tc_fence_after();
      float sc[NQ];
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + ab * N;
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        float v0[32], v1[32];
        tmem_ld_32x32b_x32(taddr + j * kHeads, v0);
        tmem_ld_32x32b_x32(taddr + j * kHeads + 32, v1);
        tmem_wait_ld();
        reg_fence_32(v0);
        reg_fence_32(v1);
        // four independent partial sums, two per paired (f32x2) FMA; weights come four at a time
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
      // this token's host row (read before the accumulator is handed back, which is
      // what lets the producer reuse the ring slot)
      int32_t hrow = -1;
      if (prefetch && P.r2h_tma) {
        const int rs = i % kR;
        if (!mbar_wait(&ctl->r2h_full[rs], (i / kR) & 1, abort, P.status)) break;
        hrow = r_smem[rs * kTileTokens + row];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tmem_empty[ab]);

      const int p = t * kTileTokens + row;
#pragma unroll
      for (int j = 0; j < NQ; ++j)
        if (p < valid[j]) {
          P.scores[(static_cast<size_t>(b) * NQ + j) * P.L_max + p] = sc[j];
          // the top-k's first radix step: count the score in its row's key window
          if (hist_on >> j & 1) {
            const int bin = sel_bin(score_key(sc[j]), ctl->hwin[e][j][0], ctl->hwin[e][j][1]);
            if (bin >= 0) red_add(P.sel_hist + static_cast<size_t>(b * NQ + j) * kSelBins + bin, 1u);
          }
        }

      if (prefetch && !(pf_cut && i + pf_tail >= n_tiles)) {
        // threshold test only; the residency test, ticket and copy happen in the
        // prefetch warps so that no global load sits on this path
        bool pass = false;
#pragma unroll
        for (int j = 0; j < NQ; ++j) pass |= (p < valid[j]) && (sc[j] > shat[j]);
        const uint32_t mask = __ballot_sync(0xffffffffu, pass);
        if (mask) {
          int n = 0;
          if (lane == 0) {
            const int head = *reinterpret_cast<volatile int *>(&ctl->queue_head[e]);
            const int room = kQueueCap - (tail - head);
            n = __popc(mask);
            n = n < room ? n : room;  // a full queue drops candidates: prefetch is best effort
          }
          n = __shfl_sync(0xffffffffu, n, 0);
          const int rank = __popc(mask & ((1u << lane) - 1));
          if (pass && rank < n) {
            ctl->queue[e][(tail + rank) % kQueueCap] = b * P.L_max + p;
            ctl->queue_h[e][(tail + rank) % kQueueCap] = hrow;
          }
          __syncwarp();
          tail += n;
          if (lane == 0 && n > 0) {
            __threadfence_block();
            *reinterpret_cast<volatile int *>(&ctl->queue_tail[e]) = tail;
          }
        }
      }
      for (int u = 0; u < kEpiGroups; ++u) next_tile(P, b, t);
    }
    if (lane == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int *>(&ctl->queue_done[e]) = 1;
    }
    if (lane == 0) ECHO_TRACE_LAST_BLOCK(26);
    if (lane == 0) ECHO_TRACE_FIRST_HERE(31);
  } else if (prefetch) {
    // ===================== prefetch copies =====================
    // prefetch warp e serves the queues of epilogue warps e, e + kPfWarps, ...
    const int pf = warp - 2 - kEpiWarps;
    const bool direct = P.reserve != nullptr;
    // reserve length (written by the recall before this kernel); once this warp has
    // seen the tickets pass it, later candidates are dropped without being read
    const int32_t res_len = direct ? __ldg(P.reserve_ctl + 1) : 0;
    bool res_full = false;
    constexpr int kQ = kEpiWarps / kPfWarps;
    int heads[kQ];
#pragma unroll
    for (int u = 0; u < kQ; ++u) heads[u] = 0;
    int turn = 0;
    uint64_t idle_since = 0;
    while (true) {
      // next queue with work, round robin; stop once every queue is done and drained
      int e = -1, tl = 0, head = 0;
      bool all_done = true, scored = true;
#pragma unroll
      for (int u = 0; u < kQ; ++u) {
        const int qi = (turn + u) % kQ;
        const int q = pf + qi * kPfWarps;
        const int done = *reinterpret_cast<volatile int *>(&ctl->queue_done[q]);
        const int tq = *reinterpret_cast<volatile int *>(&ctl->queue_tail[q]);
        scored = scored && done != 0;
        if (tq != heads[qi]) {
          if (e < 0) {
            e = q;
            tl = tq;
            head = heads[qi];
            turn = qi;
          }
          all_done = false;
        } else if (!done) {
          all_done = false;
        }
      }
      // prefetch while scoring: the epilogue warps this warp serves have scored their
      // last tiles, so what is still queued is dropped unread (nobody refills a queue
      // once its epilogue warp is done)
      if (P.pf_while_scoring && scored) break;
      if (e < 0) {
        if (all_done) break;
        const uint64_t now = globaltimer();
        if (idle_since == 0) idle_since = now;
        if (now - idle_since > kWaitLimitNs) {
          set_status(P.status, ECHO_DEV_WAIT_TIMEOUT);
          *abort = 1;
          break;
        }
        __nanosleep(200);
        continue;
      }
      volatile int *vhead = &ctl->queue_head[e];
      idle_since = 0;
      // ---- up to 32 queued tokens: host row, residency, ticket (one lane each)
      const int n = (tl - head) < 32 ? (tl - head) : 32;
      int32_t h = -1, b = 0;
      bool cand = false;
      if (lane < n) {
        const int tok = *reinterpret_cast<volatile int *>(&ctl->queue[e][(head + lane) % kQueueCap]);
        b = tok / P.L_max;
        // req_to_host is [B][L_max]: index b * L_max + p (staged with the tile when possible)
        h = P.r2h_tma ? *reinterpret_cast<volatile int *>(&ctl->queue_h[e][(head + lane) % kQueueCap])
                      : __ldg(P.req_to_host + tok);
        if (h >= 0 && h < P.n_h) {
          cand = P.host_to_gpu[h] == kInf;
        } else {
          set_status(P.status, ECHO_DEV_BAD_INDEX);
        }
      }
      head += n;  // entries are in registers: hand the slots back to the epilogue
      heads[turn] = head;
      turn = (turn + 1) % kQ;
      __syncwarp();
      if (lane == 0) *vhead = head;
      prefetch_copy_batch(P, cand, h, b, res_len, res_full);
    }
    if (lane == 0) ECHO_TRACE_LAST_HERE(27);
  }

  tc_fence_before();
  __syncthreads();
  ECHO_TRACE_LAST(25);
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


typedef CUresult (*PFN_encodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled encode_fn() {
  static std::atomic<PFN_encodeTiled> fn{nullptr};
  PFN_encodeTiled f = fn.load(std::memory_order_acquire);
  if (!f) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      f = reinterpret_cast<PFN_encodeTiled>(p);
      fn.store(f, std::memory_order_release);
    }
  }
  return f;
}

// Tensor maps of recent launches.  A map depends only on its parameters (device, data
// type, base pointer, extents, strides, box, swizzle, L2 promotion), so a launch over the
// same buffers and shape reuses the encoding instead of encoding again on the host.
struct TmapKey {
  int dev;
  CUtensorMapDataType dt;
  cuuint32_t rank;
  const void *ptr;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3];
  CUtensorMapSwizzle sw;
  CUtensorMapL2promotion l2;
};
constexpr int kTmapCache = 16;

static CUresult encode_cached(PFN_encodeTiled enc, CUtensorMap *out, CUtensorMapDataType dt, cuuint32_t rank,
                              const void *ptr, const cuuint64_t *dims, const cuuint64_t *strides,
                              const cuuint32_t *box, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  TmapKey k;
  memset(&k, 0, sizeof(k));  // padding too: keys compare bytewise
  cudaGetDevice(&k.dev);
  k.dt = dt;
  k.rank = rank;
  k.ptr = ptr;
  for (cuuint32_t i = 0; i < rank; ++i) {
    k.dims[i] = dims[i];
    k.box[i] = box[i];
    if (i + 1 < rank) k.strides[i] = strides[i];
  }
  k.sw = sw;
  k.l2 = l2;
  static std::mutex mu;
  static TmapKey keys[kTmapCache];
  static CUtensorMap maps[kTmapCache];
  static bool used[kTmapCache];
  static int next = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < kTmapCache; ++i)
      if (used[i] && memcmp(&keys[i], &k, sizeof(k)) == 0) {
        *out = maps[i];
        return CUDA_SUCCESS;
      }
  }
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(out, dt, rank, const_cast<void *>(ptr), dims, strides, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS) {
    std::lock_guard<std::mutex> lk(mu);
    keys[next] = k;
    maps[next] = *out;
    used[next] = true;
    next = (next + 1) % kTmapCache;
  }
  return r;
}

// SM count of the current device (queried once per device, so that launches
// made during stream capture issue no attribute queries)
int sm_count() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) dev = 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    n = n > 0 ? n : 1;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static size_t indexer_smem_bytes(int nq) {
  return 1024 + echo::kStages * echo::kTileBytes + 2 * (echo::kHeads * nq * echo::kDim) +
         echo::kR * echo::kRowMapBytes +
         (nq == 1 ? sizeof(echo::IndexerCtl<echo::Roles<1>::kEpiWarps>) : sizeof(echo::IndexerCtl<echo::Roles<2>::kEpiWarps>));
}

int launch_indexer(const echo_indexer_args *a, cudaStream_t stream, uint32_t *sel_hist, const int4 *sel_hint) {
  PFN_encodeTiled enc = encode_fn();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled unavailable from the driver");
    return ECHO_ECUDA;
  }
  const int nq = a->n_q;
  CUtensorMap tk, tq;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(echo::kDim), static_cast<cuuint64_t>(a->L_max),
                          static_cast<cuuint64_t>(a->B)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(echo::kDim),
                             static_cast<cuuint64_t>(a->L_max) * echo::kDim};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(echo::kDim), static_cast<cuuint32_t>(echo::kTileTokens), 1};
    CUresult r = encode_cached(enc, &tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a->k_index, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r != CUDA_SUCCESS) {
      set_error("tensor map for k_index failed (CUresult %d)", static_cast<int>(r));
      return ECHO_ECUDA;
    }
  }
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(echo::kDim),
                          static_cast<cuuint64_t>(a->B) * nq * echo::kHeads};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(echo::kDim)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(echo::kDim), static_cast<cuuint32_t>(nq * echo::kHeads)};
    CUresult r = encode_cached(enc, &tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a->q, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    if (r != CUDA_SUCCESS) {
      set_error("tensor map for q failed (CUresult %d)", static_cast<int>(r));
      return ECHO_ECUDA;
    }
  }
  // the host rows of each tile by TMA: 128 int32 per box, rows of L_max int32
  CUtensorMap tr;
  memset(&tr, 0, sizeof(tr));
  bool r2h_tma = false;
  if (a->s_hat && a->L_max % 4 == 0 && (reinterpret_cast<uintptr_t>(a->req_to_host) & 15) == 0) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(a->L_max), static_cast<cuuint64_t>(a->B)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(a->L_max) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(echo::kTileTokens), 1};
    r2h_tma = encode_cached(enc, &tr, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, a->req_to_host, dims, strides, box,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE) == CUDA_SUCCESS;
  }
  echo::IndexerParams P{};
  P.r2h_tma = r2h_tma ? 1 : 0;
  P.sel_hist = sel_hist;
  P.sel_hint = sel_hint;
  P.w = a->w;
  P.ctx_len = a->ctx_len;
  P.scores = a->scores;
  P.B = a->B;
  P.L_max = a->L_max;
  P.status = a->dev_status;
  if (a->s_hat) {
    P.s_hat = a->s_hat;
    P.req_to_host = a->req_to_host;
    P.host_to_gpu = a->pool->host_token_to_gpu;
    P.n_h = a->pool->n_h;
    P.host_kv = a->pool->host_kv;
    P.pf_while_scoring = (a->stage->flags & ECHO_PREFETCH_WHILE_SCORING) != 0;
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
  const long long tiles = static_cast<long long>(a->B) * ((a->L_max + echo::kTileTokens - 1) / echo::kTileTokens);
  if (tiles == 0) return ECHO_OK;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  const size_t smem = indexer_smem_bytes(nq);
  cudaError_t e;
  if (nq == 1) {
    static std::atomic<bool> attr1[kMaxDevices];
    if (int r = smem_limit_once(attr1, echo::indexer_kernel<1>, static_cast<int>(smem), "indexer smem attribute"))
      return r;
    echo::indexer_kernel<1><<<grid, echo::Roles<1>::kThreads, smem, stream>>>(tk, tq, tr, P);
  } else {
    static std::atomic<bool> attr2[kMaxDevices];
    if (int r = smem_limit_once(attr2, echo::indexer_kernel<2>, static_cast<int>(smem), "indexer smem attribute"))
      return r;
    echo::indexer_kernel<2><<<grid, echo::Roles<2>::kThreads, smem, stream>>>(tk, tq, tr, P);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
  return ECHO_OK;
}

int launch_indexer(const echo_indexer_args *a, cudaStream_t stream) { return launch_indexer(a, stream, nullptr, nullptr); }

}  // namespace echo_host
