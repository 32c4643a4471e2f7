// sparse_mla.cu -- sparse MLA decode over the rows the recall made resident.
//
// ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"), section 2: MLA keeps one latent
// row per token (d_c = 512, plus 64 rope dimensions) shared by all H = 128 heads, and
// the top-k rows the indexer selects feed a sparse MLA kernel (section 3.2 measures
// FlashMLA's).  With the key and value up-projections absorbed, every head h of query
// token (b, j) attends over the selected rows:
//   s_i = scale * q[b][j][h] . kv[slot_i]   (576 dims)
//   o   = sum_i softmax(s)_i * kv[slot_i][0:512],  lse = log sum_i exp(s_i)
// slot_i = out_slot[b][j][i]; entries with slot < 0 are skipped.
//
// sm_103a design (split over the selected rows, then a combine kernel):
//   one CTA (8 warps: two per TMEM lane quadrant, splitting the columns) per
//   (b, j, 128 selected rows):
//     rows   the 128 rows (576 bf16 each) copied by slot straight into shared memory
//          with cp.async (every 16-byte piece in flight at once), as nine 64-dim blocks
//          in the 128-byte swizzle: one tile that serves both products;
//     pass A  q's nine 64-dim blocks (128 heads each) stream in by TMA through a
//          5-stage ring (a stage is refilled once the MMAs of the block before the
//          current one are done); four tcgen05 MMAs per block (kind::f16, bf16 x
//          bf16 -> fp32, M = 128 heads, N = 128 rows, K = 16) accumulate S in TMEM
//          columns 0..127;
//     softmax  two threads per head, 64 columns each (maxima and sums exchanged
//          through shared memory): S from TMEM, scale, mask, max, exp, sum;
//          P (bf16) into shared memory (where the q ring was) as the next MMA's
//          K-major operand;
//     pass B  O += P . V on tcgen05 with V the first eight blocks of the same row tile
//          read as an MN-major operand, two N = 256 halves of 8 MMAs into all 512 TMEM
//          columns (S has been consumed);
//     partial O divided by the split's sum, in fp16, stored dims-major (a warp writes
//          32 heads of one dim: coalesced), max and sum per head;
//   combine: per (b, j) and 16-dim slice, the split weights once per block in shared
//          memory, 16-byte partial loads, the result transposed for float4 stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "echo_common.cuh"

ECHO_TRACE_UNIT(sparse_mla)

namespace echo {

constexpr int kMlaHeads = 128;                   // MMA M
constexpr int kMlaDqk = kKvElems;                // 576
constexpr int kMlaDv = 512;
constexpr int kMlaBlocks = kMlaDqk / 64;         // 9 swizzled 64-dim blocks
constexpr int kMlaSplit = 128;                   // selected rows per CTA (MMA N of pass A)
constexpr int kMlaMaxK = 8192;                   // the largest k the C ABI accepts
constexpr int kMlaThreads = 256;
constexpr int kMlaStages = 5;                    // ring of q blocks
constexpr int kMlaGroups = 3;                    // commit groups of the row gather
constexpr int kMlaGroupBlocks = 3;               // 64-dim blocks per group
static_assert(kMlaGroups * kMlaGroupBlocks == 576 / 64 && kMlaGroups == 3, "the gather's waits cover 3 groups");
constexpr uint32_t kMlaTile = 128 * 128;         // 128 rows (or heads) x one 64-dim block: 16 KB
constexpr uint32_t kMlaRowsBytes = kMlaBlocks * kMlaTile;        // the 128 rows: 144 KB
constexpr uint32_t kMlaVHalf = 4 * kMlaTile;                     // 256 value dims of the 128 rows
constexpr uint32_t kMlaRingBytes = kMlaStages * kMlaTile;
constexpr uint32_t kMlaPBytes = 2 * kMlaTile;                    // P: 128 heads x 128 rows bf16
constexpr uint32_t kMlaTmemCols = 512;

struct MlaParams {
  const uint16_t *gpu_kv;    // [n_g][576]
  const int32_t *out_slot;   // [B][n_q][k]
  int32_t n_g, n_q, k, nsplit;
  float scale;
  __half *part_o;            // [units][512][128] (dims-major), divided by the split's sum
  float *part_ml;            // [units][2][128]: max, sum
  int32_t *status;
};

// Instruction descriptor of tcgen05.mma kind::f16: D fp32, A = B = bf16, A K-major,
// B K-major (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// MN-major operand in the 128-byte swizzle: 64 elements (128 bytes) along N per
// row of the tile, rows (the K dimension) 128 bytes apart in 1024-byte groups of 8;
// lbo = distance between consecutive 64-element groups along N, sbo = between
// consecutive 8-row groups along K.
__device__ __forceinline__ uint64_t mnmajor_sw128_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// generic-proxy shared-memory writes -> visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// A wait the whole CTA agrees on: thread 0 waits (bounded), a barrier hands the
// outcome to every thread, so that no thread leaves a loop the others stay in.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t parity, volatile int *abort, int32_t *status,
                                         int *flag) {
  if (threadIdx.x == 0) *flag = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  __syncthreads();
  const bool ok = *reinterpret_cast<volatile int *>(flag) != 0;
  __syncthreads();  // the flag may be rewritten by the next wait
  return ok;
}

// 16-byte asynchronous copy global -> shared (zero-filled when src_bytes = 0)
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_q, const MlaParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *rows_smem = smem;                                // 9 blocks x 128 rows x 128 B
  uint8_t *ring = rows_smem + kMlaRowsBytes;                // 5 stages of q blocks
  uint8_t *p_smem = ring;                                   // after pass A: 2 blocks x 128 heads x 128 B
  // barriers: q landed per stage, MMAs of the stage's block done per stage, pass B, drain
  // (a stage's barriers never run more than one phase ahead of their waiter)
  constexpr int kBarMma = kMlaStages, kBarPv = 2 * kMlaStages, kBarDrain = 2 * kMlaStages + 1;
  constexpr int kNumBars = 2 * kMlaStages + 2;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ring + kMlaRingBytes);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
  int32_t *s_slot = reinterpret_cast<int32_t *>(tmem_slot + 4);       // [128]
  int *abort_flag = s_slot + kMlaSplit;
  int *wait_flag = abort_flag + 1;
  volatile int *abort = abort_flag;

  const int unit = blockIdx.x;
  const int bj = unit / P.nsplit, split = unit % P.nsplit;
  const int row0 = split * kMlaSplit;
  const int nrows = min(kMlaSplit, P.k - row0);
  const int warp = threadIdx.x >> 5;
  const int h = (warp & 3) * 32 + (threadIdx.x & 31);  // head = TMEM lane (the warp's quadrant)
  const int half = warp >> 2;                           // which half of the columns
  ECHO_TRACE_FIRST(0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < kMlaSplit; i += kMlaThreads) {
    int32_t s = i < nrows ? __ldg(P.out_slot + static_cast<size_t>(bj) * P.k + row0 + i) : -1;
    if (s >= P.n_g) {
      set_status(P.status, ECHO_DEV_BAD_INDEX);
      s = -1;
    }
    s_slot[i] = s;
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kMlaTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t trow = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
  // q's first blocks by TMA; the rows by cp.async, every piece in flight together, issued
  // block by block (64 dims of all 128 rows) in kMlaGroups commit groups so that pass A
  // starts on the first blocks while the later ones are still on their way
  if (threadIdx.x == 0)
    for (int d = 0; d < kMlaStages; ++d) {
      mbar_arrive_expect_tx(&bars[d], kMlaTile);
      tma_load_2d(ring + d * kMlaTile, &tmap_q, &bars[d], d * 64, bj * kMlaHeads);
    }
  {
    const int4 *kv = reinterpret_cast<const int4 *>(P.gpu_kv);
#pragma unroll
    for (int g = 0; g < kMlaGroups; ++g) {
#pragma unroll
      for (int blk = g * kMlaGroupBlocks; blk < (g + 1) * kMlaGroupBlocks; ++blk) {
#pragma unroll
        for (int t = threadIdx.x; t < kMlaSplit * 8; t += kMlaThreads) {
          const int r = t >> 3, c = t & 7;  // a warp copies 128 bytes of each of 4 rows
          const int32_t slot = s_slot[r];
          cp_async16(rows_smem + blk * kMlaTile + r * 128 + ((c ^ (r & 7)) << 4),
                     kv + static_cast<size_t>(slot >= 0 ? slot : 0) * kKvChunks + blk * 8 + c, slot >= 0 ? 16u : 0u);
        }
      }
      cp_async_commit();
    }
  }
  bool ok = true;
  bool issued = false;  // thread 0 issued tcgen05 work (drained on a failure)

  // ===== pass A: S = q . rows^T, one 64-dim block of q per ring stage (thread 0), each
  // group of row blocks as soon as every thread's copies of it have landed =====
  constexpr uint32_t kIdescA = idesc_bf16_f32(kMlaHeads, kMlaSplit, 0);
  int waited = 0;  // (thread 0) blocks whose MMAs were seen done, in order
#pragma unroll
  for (int g = 0; g < kMlaGroups; ++g) {
    if (g == 0) cp_async_wait_group<kMlaGroups - 1>();
    else if (g == 1) cp_async_wait_group<kMlaGroups - 2>();
    else cp_async_wait_all();
    fence_async_smem();
    __syncthreads();
    if (g == kMlaGroups - 1) ECHO_TRACE_LAST(1);
    if (threadIdx.x != 0 || !ok) continue;
    tc_fence_after();
    const uint32_t ra = smem_u32(rows_smem);
    for (int d = g * kMlaGroupBlocks; d < (g + 1) * kMlaGroupBlocks; ++d) {
      const int st = d % kMlaStages;
      if (!mbar_wait(&bars[st], (d / kMlaStages) & 1, abort, P.status)) {  // q's block d landed
        ok = false;
        break;
      }
      const uint32_t qa = smem_u32(ring + st * kMlaTile);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_bf16(tmem, kmajor_sw128_desc(qa + kk * 32), kmajor_sw128_desc(ra + d * kMlaTile + kk * 32), kIdescA,
                 (d | kk) != 0);
      mma_commit(&bars[kBarMma + st]);
      issued = true;
      // refill the stage of block d - 1 (its MMAs ran while these were queued) with
      // block d - 1 + kMlaStages
      const int nb = d - 1 + kMlaStages;
      if (d >= 1 && nb < kMlaBlocks) {
        const int pd = d - 1;
        if (!mbar_wait(&bars[kBarMma + pd % kMlaStages], (pd / kMlaStages) & 1, abort, P.status)) {
          ok = false;
          break;
        }
        waited = d;
        const int s2 = nb % kMlaStages;
        mbar_arrive_expect_tx(&bars[s2], kMlaTile);
        tma_load_2d(ring + s2 * kMlaTile, &tmap_q, &bars[s2], nb * 64, bj * kMlaHeads);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (; ok && waited < kMlaBlocks; ++waited)  // every pass-A MMA is done
      if (!mbar_wait(&bars[kBarMma + waited % kMlaStages], (waited / kMlaStages) & 1, abort, P.status)) ok = false;
    *wait_flag = ok ? 1 : 0;
  }
  __syncthreads();
  ok = *reinterpret_cast<volatile int *>(wait_flag) != 0;
  __syncthreads();
  ECHO_TRACE_LAST(2);

  // ===== softmax over this CTA's rows: two threads per head, 64 columns each =====
  float *red = reinterpret_cast<float *>(ring + 2 * kMlaTile);  // [2][2][128] maxima, sums (free stages)
  float l_sum = 0.f;
  if (ok) {
    tc_fence_after();
    const int cb = half * 64;
    float s[64];
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) {
      float v[32];
      tmem_ld_32x32b_x32(trow + cb + c2 * 32, v);
      tmem_wait_ld();
      reg_fence_32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c2 * 32 + i] = v[i];
    }
    float mh = -INFINITY;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      s[i] = s_slot[cb + i] >= 0 ? s[i] * P.scale : -INFINITY;
      mh = fmaxf(mh, s[i]);
    }
    red[half * kMlaHeads + h] = mh;
    __syncthreads();
    const float m = fmaxf(red[h], red[kMlaHeads + h]);
    // P = exp(s - m) in bf16 (K-major operand: head row h, this half's 64 rows = one block)
    float lh = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = m == -INFINITY ? 0.f : __expf(s[c8 * 8 + 2 * u] - m);
        const float b = m == -INFINITY ? 0.f : __expf(s[c8 * 8 + 2 * u + 1] - m);
        lh += a + b;
        const __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
        w[u] = *reinterpret_cast<const uint32_t *>(&pr);
      }
      *reinterpret_cast<uint4 *>(p_smem + half * kMlaTile + h * 128 + ((c8 ^ (h & 7)) << 4)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    red[2 * kMlaHeads + half * kMlaHeads + h] = lh;
    __syncthreads();
    l_sum = red[2 * kMlaHeads + h] + red[3 * kMlaHeads + h];
    if (half == 0) {
      P.part_ml[static_cast<size_t>(unit) * 2 * kMlaHeads + h] = m;
      P.part_ml[static_cast<size_t>(unit) * 2 * kMlaHeads + kMlaHeads + h] = l_sum;
    }
  }
  tc_fence_before();
  fence_async_smem();
  __syncthreads();
  ECHO_TRACE_LAST(3);

  // ===== pass B: O += P . V (V = the row tile's first 512 dims, read along the rows:
  // MN-major), two halves of 256 dims =====
  constexpr uint32_t kIdescB = idesc_bf16_f32(kMlaHeads, 256, 1);
  if (ok && threadIdx.x == 0) {
    tc_fence_after();
    const uint32_t pa = smem_u32(p_smem);
    for (int half = 0; half < 2; ++half) {
      const uint32_t va = smem_u32(rows_smem + half * kMlaVHalf);
#pragma unroll
      for (int kk = 0; kk < kMlaSplit / 16; ++kk)
        mma_bf16(tmem + half * 256, kmajor_sw128_desc(pa + (kk >> 2) * kMlaTile + (kk & 3) * 32),
                 mnmajor_sw128_desc(va + kk * 16 * 128, kMlaTile, 1024), kIdescB, kk > 0);
    }
    mma_commit(&bars[kBarPv]);
    issued = true;
  }
  if (ok && !cta_wait(&bars[kBarPv], 0, abort, P.status, wait_flag)) ok = false;
  ECHO_TRACE_LAST(4);

  // ===== partial O of this CTA's rows, dims-major: a warp stores 32 heads of one dim
  // (coalesced); the two warps of a lane quadrant take 256 dims each =====
  if (ok) {
    tc_fence_after();
    __half *dst = P.part_o + static_cast<size_t>(unit) * kMlaDv * kMlaHeads + h;
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll 1
    for (int c32 = 0; c32 < kMlaDv / 2 / 32; ++c32) {
      const int d0 = half * (kMlaDv / 2) + c32 * 32;
      float v[32];
      tmem_ld_32x32b_x32(trow + d0, v);
      tmem_wait_ld();
      reg_fence_32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[static_cast<size_t>(d0 + i) * kMlaHeads] = __float2half_rn(v[i] * inv);
    }
  }
  if (!ok && threadIdx.x == 0) {
    // a wait gave up: let the q copy and every MMA this CTA started finish before it
    // frees TMEM and exits (one commit after them all, waited on with a limit)
    for (int st = 0; st < kMlaStages; ++st) {  // q copies that may still be in flight
      const uint64_t t2 = globaltimer();
      while (!mbar_try_wait(&bars[st], 0) && globaltimer() - t2 < kWaitLimitNs) {
      }
    }
    if (issued) {
      mma_commit(&bars[kBarDrain]);
      const uint64_t t1 = globaltimer();
      while (!mbar_try_wait(&bars[kBarDrain], 0) && globaltimer() - t1 < kWaitLimitNs) {
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  ECHO_TRACE_LAST(5);
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
}

// o = sum_s w_s l_s o_s / sum_s w_s l_s (o_s the split's normalised partial),
// w_s = exp(m_s - max_s m_s); lse = max + log(sum).  Block (bj, slice of 16 dims), 256
// threads: thread (dim d, group g of 8 heads) reads 16 bytes of one split's partial per
// load (16 threads cover a dim's 128 heads: 256 contiguous bytes), sixteen splits' loads
// issued before the weights are known.  The split weights of all 128 heads are computed
// once per block into shared memory; the result tile is transposed in shared memory so
// each head's 16 dims leave as four float4 stores.
constexpr int kCombDims = 16;
constexpr int kCombThreads = 256;
constexpr int kCombChunk = 16;                      // splits whose loads are in flight together
constexpr int kCombMaxSplits = kMlaMaxK / kMlaSplit;

__global__ void __launch_bounds__(kCombThreads) sparse_mla_combine_kernel(const __half *part_o, const float *part_ml,
                                                                           int nsplit, float *out, float *lse) {
  __shared__ __align__(16) float w_s[kCombMaxSplits][kMlaHeads];
  __shared__ __align__(16) float o_s[kCombDims][kMlaHeads + 4];
  __shared__ float il_s[kMlaHeads];
  const int bj = blockIdx.x, d0 = blockIdx.y * kCombDims, t = threadIdx.x;
  const int d = t / 16, h8 = 8 * (t % 16);
  ECHO_TRACE_FIRST(6);
  const uint4 *src = reinterpret_cast<const uint4 *>(part_o + (static_cast<size_t>(bj) * nsplit * kMlaDv + d0 + d) *
                                                                   kMlaHeads + h8);
  const size_t split_stride = static_cast<size_t>(kMlaDv) * kMlaHeads / 8;   // in uint4
  uint4 v[kCombChunk];
#pragma unroll
  for (int q = 0; q < kCombChunk; ++q)
    v[q] = q < nsplit ? __ldcs(src + q * split_stride) : make_uint4(0u, 0u, 0u, 0u);
  if (t < kMlaHeads) {
    // head t: the maximum over the splits, then each split's weight w_s l_s
    const float *ml = part_ml + static_cast<size_t>(bj) * nsplit * 2 * kMlaHeads + t;
    float M = -INFINITY;
    for (int s0 = 0; s0 < nsplit; s0 += kCombChunk) {
      float m[kCombChunk];
#pragma unroll
      for (int q = 0; q < kCombChunk; ++q) m[q] = s0 + q < nsplit ? ml[(s0 + q) * 2 * kMlaHeads] : -INFINITY;
#pragma unroll
      for (int q = 0; q < kCombChunk; ++q) M = fmaxf(M, m[q]);
    }
    float L = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += kCombChunk) {
      float m[kCombChunk], l[kCombChunk];
#pragma unroll
      for (int q = 0; q < kCombChunk; ++q) {
        const bool in = s0 + q < nsplit;
        m[q] = in ? ml[(s0 + q) * 2 * kMlaHeads] : -INFINITY;
        l[q] = in ? ml[(s0 + q) * 2 * kMlaHeads + kMlaHeads] : 0.f;
      }
#pragma unroll
      for (int q = 0; q < kCombChunk; ++q) {
        if (s0 + q < nsplit) {
          const float w = M == -INFINITY ? 0.f : __expf(m[q] - M) * l[q];
          w_s[s0 + q][t] = w;
          L += w;
        }
      }
    }
    il_s[t] = L > 0.f ? 1.f / L : 0.f;
    if (blockIdx.y == 0) lse[static_cast<size_t>(bj) * kMlaHeads + t] = M == -INFINITY ? -INFINITY : M + logf(L);
  }
  __syncthreads();
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  for (int s0 = 0;; s0 += kCombChunk) {
#pragma unroll
    for (int q = 0; q < kCombChunk; ++q) {
      if (s0 + q < nsplit) {
        const float4 wa = *reinterpret_cast<const float4 *>(&w_s[s0 + q][h8]);
        const float4 wb = *reinterpret_cast<const float4 *>(&w_s[s0 + q][h8 + 4]);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&v[q].x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&v[q].y));
        const float2 f2 = __half22float2(*reinterpret_cast<const __half2 *>(&v[q].z));
        const float2 f3 = __half22float2(*reinterpret_cast<const __half2 *>(&v[q].w));
        acc[0] = fmaf(wa.x, f0.x, acc[0]);
        acc[1] = fmaf(wa.y, f0.y, acc[1]);
        acc[2] = fmaf(wa.z, f1.x, acc[2]);
        acc[3] = fmaf(wa.w, f1.y, acc[3]);
        acc[4] = fmaf(wb.x, f2.x, acc[4]);
        acc[5] = fmaf(wb.y, f2.y, acc[5]);
        acc[6] = fmaf(wb.z, f3.x, acc[6]);
        acc[7] = fmaf(wb.w, f3.y, acc[7]);
      }
    }
    if (s0 + kCombChunk >= nsplit) break;
#pragma unroll
    for (int q = 0; q < kCombChunk; ++q)
      v[q] = s0 + kCombChunk + q < nsplit ? __ldcs(src + (s0 + kCombChunk + q) * split_stride)
                                          : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) o_s[d][h8 + i] = acc[i] * il_s[h8 + i];
  __syncthreads();
  // out[bj][h][d0 .. d0 + 16): 128 heads x 4 float4
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int f = t + kCombThreads * r, h = f / 4, c = 4 * (f % 4);
    const float4 o = make_float4(o_s[c][h], o_s[c + 1][h], o_s[c + 2][h], o_s[c + 3][h]);
    *reinterpret_cast<float4 *>(out + (static_cast<size_t>(bj) * kMlaHeads + h) * kMlaDv + d0 + c) = o;
  }
  ECHO_TRACE_LAST(7);
}

}  // namespace echo

// ---------------------------------------------------------------------------
// host launcher
// ---------------------------------------------------------------------------
namespace echo_host {

typedef CUresult (*PFN_encodeTiledM)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                     CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);

static PFN_encodeTiledM encode_fn_m() {
  static PFN_encodeTiledM fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiledM>(p);
  }
  return fn;
}

size_t mla_workspace_bytes(int32_t B, int32_t n_q, int32_t k) {
  const size_t nsplit = (static_cast<size_t>(k) + echo::kMlaSplit - 1) / echo::kMlaSplit;
  const size_t units = static_cast<size_t>(B) * n_q * nsplit;
  return units * echo::kMlaHeads * (echo::kMlaDv * sizeof(__half) + 2 * sizeof(float));
}

int launch_sparse_mla(const echo_mla_args *a, cudaStream_t stream) {
  PFN_encodeTiledM enc = encode_fn_m();
  if (!enc) {
    set_error("cuTensorMapEncodeTiled unavailable from the driver");
    return ECHO_ECUDA;
  }
  CUtensorMap tq;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(echo::kMlaDqk),
                        static_cast<cuuint64_t>(a->B) * a->n_q * echo::kMlaHeads};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(echo::kMlaDqk) * 2};
  cuuint32_t box[2] = {64, static_cast<cuuint32_t>(echo::kMlaHeads)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a->q), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("tensor map for the MLA queries failed (CUresult %d)", static_cast<int>(r));
    return ECHO_ECUDA;
  }
  echo::MlaParams P{};
  P.gpu_kv = a->gpu_kv;
  P.out_slot = a->out_slot;
  P.n_g = a->n_g;
  P.n_q = a->n_q;
  P.k = a->k;
  P.nsplit = (a->k + echo::kMlaSplit - 1) / echo::kMlaSplit;
  if (P.nsplit > echo::kCombMaxSplits) {
    set_error("sparse MLA: k above %d", echo::kMlaMaxK);
    return ECHO_EINVAL;
  }
  P.scale = a->scale;
  const size_t units = static_cast<size_t>(a->B) * a->n_q * P.nsplit;
  P.part_o = reinterpret_cast<__half *>(a->workspace);
  P.part_ml = reinterpret_cast<float *>(P.part_o + units * echo::kMlaHeads * echo::kMlaDv);
  P.status = a->dev_status;
  static_assert(echo::kMlaPBytes <= echo::kMlaRingBytes, "P lives in the q ring");
  const size_t smem = 1024 + echo::kMlaRowsBytes + echo::kMlaRingBytes + (2 * echo::kMlaStages + 2) * 8 + 16 +
                      echo::kMlaSplit * sizeof(int32_t) + 16;
  static std::atomic<bool> attr[kMaxDevices];
  if (int rr = smem_limit_once(attr, echo::sparse_mla_kernel, static_cast<int>(smem), "sparse MLA smem attribute"))
    return rr;
  echo::sparse_mla_kernel<<<static_cast<unsigned>(units), echo::kMlaThreads, smem, stream>>>(tq, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse MLA launch");
  // an ordinary launch: as a programmatic dependent launch the merge started sooner
  // but ran slower (its blocks were placed while the main kernel held the SMs)
  const dim3 cgrid(static_cast<unsigned>(a->B * a->n_q), echo::kMlaDv / echo::kCombDims);
  echo::sparse_mla_combine_kernel<<<cgrid, echo::kCombThreads, 0, stream>>>(P.part_o, P.part_ml, P.nsplit, a->out,
                                                                            a->lse);
  e = cudaGetLastError();
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "sparse MLA combine launch");
}

}  // namespace echo_host
