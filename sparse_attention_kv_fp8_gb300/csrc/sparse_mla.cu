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
//   one CTA (4 warps) per (b, j, 128 selected rows):
//     q    128 heads x 576 bf16 by TMA into nine 128-byte-swizzled 64-dim blocks;
//     pass A  the 128 rows gathered 16 at a time (16-byte loads by slot, written in the
//          same swizzled layout, double buffered) and S = q . rows^T on tcgen05
//          (kind::f16, bf16 x bf16 -> fp32, M = 128 heads, N = 16 rows, K = 576) into
//          TMEM columns 0..127;
//     softmax  one thread per head: its S row from TMEM, scale, mask, max, exp, sum;
//          P (bf16) into shared memory as the next MMA's K-major operand;
//     pass B  the rows gathered again (512 dims; they are in L2) and O += P . V on
//          tcgen05 with V as an MN-major operand (the same swizzled tile, read along
//          the rows), two N = 256 MMAs per 16 rows into all 512 TMEM columns;
//     partial O, max and sum per head to a workspace;
//   combine: per (b, j, head) the splits' partials merged with their maxima.
#include <cuda_bf16.h>

#include "echo_common.cuh"

namespace echo {

constexpr int kMlaHeads = 128;                   // MMA M
constexpr int kMlaDqk = kKvElems;                // 576
constexpr int kMlaDv = 512;
constexpr int kMlaBlocks = kMlaDqk / 64;         // 9 swizzled 64-dim blocks
constexpr int kMlaSplit = 128;                   // selected rows per CTA
constexpr int kMlaChunk = 16;                    // rows per gathered chunk
constexpr int kMlaChunks = kMlaSplit / kMlaChunk;
constexpr int kMlaThreads = 128;
constexpr uint32_t kMlaQBytes = kMlaBlocks * kMlaHeads * 128;    // 147456
constexpr uint32_t kMlaBlockBytes = kMlaChunk * 128;            // one 64-dim block of a chunk: 2048
constexpr uint32_t kMlaChunkBytes = kMlaBlocks * kMlaBlockBytes;  // 18432
constexpr uint32_t kMlaPBytes = 2 * kMlaHeads * 128;             // 128 heads x 128 rows bf16
constexpr uint32_t kMlaTmemCols = 512;

struct MlaParams {
  const uint16_t *gpu_kv;    // [n_g][576]
  const int32_t *out_slot;   // [B][n_q][k]
  int32_t n_g, n_q, k, nsplit;
  float scale;
  float *part_o;             // [units][128][512]
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

// Gathers rows [r0, r0 + 16) of this CTA's selection (the slots in s_slot) into a
// chunk buffer: block d (64 dims) of row r at d * 2048 + r * 128, its 16-byte chunks
// swizzled by r % 8.  Rows past the selection or with no slot are zero.
template <int NB>
__device__ __forceinline__ void gather_chunk(uint8_t *buf, const int4 *kv, const int32_t *s_slot, int r0, int nrows) {
  constexpr int kPer = NB * 8;  // 16-byte chunks per row
  for (int t = threadIdx.x; t < kMlaChunk * kPer; t += kMlaThreads) {
    const int r = t / kPer, ch = t % kPer;
    const int row = r0 + r;
    const int32_t slot = row < nrows ? s_slot[row] : -1;
    int4 v = make_int4(0, 0, 0, 0);
    if (slot >= 0) v = __ldg(kv + static_cast<size_t>(slot) * kKvChunks + ch);
    const int blk = ch >> 3, c = ch & 7;
    *reinterpret_cast<int4 *>(buf + blk * kMlaBlockBytes + r * 128 + ((c ^ (r & 7)) << 4)) = v;
  }
}

__global__ void __launch_bounds__(kMlaThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_q, const MlaParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *q_smem = smem;                                   // 9 blocks x 128 heads x 128 B
  uint8_t *kv_smem = q_smem + kMlaQBytes;                   // 2 chunk buffers
  uint8_t *p_smem = kv_smem + 2 * kMlaChunkBytes;           // 2 blocks x 128 heads x 128 B
  uint64_t *bars = reinterpret_cast<uint64_t *>(p_smem + kMlaPBytes);  // q_full, mma[2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
  int32_t *s_slot = reinterpret_cast<int32_t *>(tmem_slot + 4);       // [128]
  int *abort_flag = s_slot + kMlaSplit;
  int *wait_flag = abort_flag + 1;
  volatile int *abort = abort_flag;

  const int unit = blockIdx.x;
  const int bj = unit / P.nsplit, split = unit % P.nsplit;
  const int row0 = split * kMlaSplit;
  const int nrows = min(kMlaSplit, P.k - row0);
  const int nch = (nrows + kMlaChunk - 1) / kMlaChunk;
  const int h = threadIdx.x;  // head = TMEM lane
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
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
  const int4 *kv = reinterpret_cast<const int4 *>(P.gpu_kv);

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[0], kMlaQBytes);
    for (int blk = 0; blk < kMlaBlocks; ++blk)
      tma_load_2d(q_smem + blk * kMlaHeads * 128, &tmap_q, &bars[0], blk * 64, bj * kMlaHeads);
  }
  bool ok = true;
  uint32_t mma_uses[2] = {0, 0};  // commits so far on each chunk buffer's barrier

  // ===== pass A: S[:, rows] = q . rows^T =====
  constexpr uint32_t kIdescA = idesc_bf16_f32(kMlaHeads, kMlaChunk, 0);
  for (int c = 0; c < nch && ok; ++c) {
    const int bi = c & 1;
    uint8_t *buf = kv_smem + bi * kMlaChunkBytes;
    // the buffer's previous MMAs are done before it is overwritten
    if (mma_uses[bi] > 0 && !cta_wait(&bars[1 + bi], (mma_uses[bi] - 1) & 1, abort, P.status, wait_flag)) {
      ok = false;
      break;
    }
    gather_chunk<kMlaBlocks>(buf, kv, s_slot, c * kMlaChunk, nrows);
    fence_async_smem();
    if (c == 0 && !cta_wait(&bars[0], 0, abort, P.status, wait_flag)) {  // q landed (also the barrier)
      ok = false;
      break;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t qa = smem_u32(q_smem), ba = smem_u32(buf);
#pragma unroll 4
      for (int kk = 0; kk < kMlaBlocks * 4; ++kk) {
        const uint32_t blk = kk >> 2, kin = (kk & 3) * 32;
        mma_bf16(tmem + c * kMlaChunk, kmajor_sw128_desc(qa + blk * kMlaHeads * 128 + kin),
                 kmajor_sw128_desc(ba + blk * kMlaBlockBytes + kin), kIdescA, kk > 0);
      }
      mma_commit(&bars[1 + bi]);
    }
    ++mma_uses[bi];
  }
  // every pass-A MMA has completed once both buffers' last commits have
  for (int bi = 0; bi < 2 && ok; ++bi)
    if (mma_uses[bi] > 0 && !cta_wait(&bars[1 + bi], (mma_uses[bi] - 1) & 1, abort, P.status, wait_flag))
      ok = false;

  // ===== softmax over this CTA's rows, one thread per head =====
  float m = -INFINITY, l = 0.f;
  if (ok) {
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float s[kMlaSplit];
#pragma unroll
    for (int c4 = 0; c4 < kMlaSplit / 32; ++c4) {
      float v[32];
      tmem_ld_32x32b_x32(trow + c4 * 32, v);
      tmem_wait_ld();
      reg_fence_32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c4 * 32 + i] = v[i];
    }
#pragma unroll
    for (int i = 0; i < kMlaSplit; ++i) {
      s[i] = s_slot[i] >= 0 ? s[i] * P.scale : -INFINITY;
      m = fmaxf(m, s[i]);
    }
    // P = exp(s - m) in bf16 (K-major operand: head row h, rows in two 64-row blocks)
#pragma unroll
    for (int c8 = 0; c8 < kMlaSplit / 8; ++c8) {
      uint32_t w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = m == -INFINITY ? 0.f : __expf(s[c8 * 8 + 2 * u] - m);
        const float b = m == -INFINITY ? 0.f : __expf(s[c8 * 8 + 2 * u + 1] - m);
        l += a + b;
        const __nv_bfloat162 pr = __floats2bfloat162_rn(a, b);
        w[u] = *reinterpret_cast<const uint32_t *>(&pr);
      }
      const int blk = c8 >> 3, c = c8 & 7;
      *reinterpret_cast<uint4 *>(p_smem + blk * kMlaHeads * 128 + h * 128 + ((c ^ (h & 7)) << 4)) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
    P.part_ml[static_cast<size_t>(unit) * 2 * kMlaHeads + h] = m;
    P.part_ml[static_cast<size_t>(unit) * 2 * kMlaHeads + kMlaHeads + h] = l;
  }
  tc_fence_before();
  fence_async_smem();
  __syncthreads();

  // ===== pass B: O += P[:, rows] . V[rows] (V read along the rows: MN-major) =====
  constexpr uint32_t kIdescB = idesc_bf16_f32(kMlaHeads, 256, 1);
  for (int c = 0; c < nch && ok; ++c) {
    const int bi = c & 1;
    uint8_t *buf = kv_smem + bi * kMlaChunkBytes;
    if (mma_uses[bi] > 0 && !cta_wait(&bars[1 + bi], (mma_uses[bi] - 1) & 1, abort, P.status, wait_flag)) {
      ok = false;
      break;
    }
    gather_chunk<kMlaDv / 64>(buf, kv, s_slot, c * kMlaChunk, nrows);
    fence_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t pa = smem_u32(p_smem) + (c >> 2) * kMlaHeads * 128 + (c & 3) * 32;
      const uint32_t va = smem_u32(buf);
#pragma unroll
      for (int nh = 0; nh < 2; ++nh)
        mma_bf16(tmem + nh * 256, kmajor_sw128_desc(pa),
                 mnmajor_sw128_desc(va + nh * 4 * kMlaBlockBytes, kMlaBlockBytes, 1024), kIdescB, c > 0);
      mma_commit(&bars[1 + bi]);
    }
    ++mma_uses[bi];
  }
  for (int bi = 0; bi < 2 && ok; ++bi)
    if (mma_uses[bi] > 0 && !cta_wait(&bars[1 + bi], (mma_uses[bi] - 1) & 1, abort, P.status, wait_flag))
      ok = false;

  // ===== partial O of this CTA's rows =====
  if (ok) {
    tc_fence_after();
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float4 *dst = reinterpret_cast<float4 *>(P.part_o + (static_cast<size_t>(unit) * kMlaHeads + h) * kMlaDv);
    for (int c32 = 0; c32 < kMlaDv / 32; ++c32) {
      float v[32];
      tmem_ld_32x32b_x32(trow + c32 * 32, v);
      tmem_wait_ld();
      reg_fence_32(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[c32 * 8 + i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    }
  }
  if (!ok && threadIdx.x == 0) {
    // a wait gave up: let the copies and MMAs this CTA started finish before it exits
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&bars[0], 0) && globaltimer() - t0 < kWaitLimitNs) {
    }
    for (int bi = 0; bi < 2; ++bi)
      if (mma_uses[bi] > 0) {
        const uint64_t t1 = globaltimer();
        while (!mbar_try_wait(&bars[1 + bi], (mma_uses[bi] - 1) & 1) && globaltimer() - t1 < kWaitLimitNs) {
        }
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kMlaTmemCols);
  }
}

// o = sum_s w_s O_s / sum_s w_s l_s, w_s = exp(m_s - max_s m_s); lse = max + log(sum)
__global__ void sparse_mla_combine_kernel(const float *part_o, const float *part_ml, int nsplit, int n_rows,
                                          float *out, float *lse) {
  const int r = blockIdx.x;  // (b, j, head)
  if (r >= n_rows) return;
  const int bj = r / kMlaHeads, h = r % kMlaHeads;
  __shared__ float wts[64];
  __shared__ float s_inv;
  if (threadIdx.x == 0) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[(static_cast<size_t>(bj) * nsplit + s) * 2 * kMlaHeads + h]);
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t base = (static_cast<size_t>(bj) * nsplit + s) * 2 * kMlaHeads;
      const float ms = part_ml[base + h];
      const float w = M == -INFINITY ? 0.f : __expf(ms - M);
      wts[s] = w;
      L += w * part_ml[base + kMlaHeads + h];
    }
    s_inv = L > 0.f ? 1.f / L : 0.f;
    lse[r] = M == -INFINITY ? -INFINITY : M + logf(L);
  }
  __syncthreads();
  for (int d = threadIdx.x; d < kMlaDv; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s)
      acc += wts[s] * part_o[((static_cast<size_t>(bj) * nsplit + s) * kMlaHeads + h) * kMlaDv + d];
    out[static_cast<size_t>(r) * kMlaDv + d] = acc * s_inv;
  }
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
  return units * echo::kMlaHeads * (echo::kMlaDv + 2) * sizeof(float);
}

int mla_max_splits() { return 64; }

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
  P.scale = a->scale;
  const size_t units = static_cast<size_t>(a->B) * a->n_q * P.nsplit;
  P.part_o = reinterpret_cast<float *>(a->workspace);
  P.part_ml = P.part_o + units * echo::kMlaHeads * echo::kMlaDv;
  P.status = a->dev_status;
  const size_t smem = 1024 + echo::kMlaQBytes + 2 * echo::kMlaChunkBytes + echo::kMlaPBytes + 64 +
                      echo::kMlaSplit * sizeof(int32_t) + 32;
  static bool attr[64] = {false};
  if (int rr = smem_limit_once(attr, echo::sparse_mla_kernel, static_cast<int>(smem), "sparse MLA smem attribute"))
    return rr;
  echo::sparse_mla_kernel<<<static_cast<unsigned>(units), echo::kMlaThreads, smem, stream>>>(tq, P);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "sparse MLA launch");
  const int rows = a->B * a->n_q * echo::kMlaHeads;
  echo::sparse_mla_combine_kernel<<<rows, 128, 0, stream>>>(P.part_o, P.part_ml, P.nsplit, rows, a->out, a->lse);
  e = cudaGetLastError();
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "sparse MLA combine launch");
}

}  // namespace echo_host
