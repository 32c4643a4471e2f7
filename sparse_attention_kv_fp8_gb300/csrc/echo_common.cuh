// echo_common.cuh -- device helpers shared by the sm_103a kernels of the ECHO
// decode step: status bits, bounded waits, and thin inline-PTX wrappers for
// mbarrier, TMA (cp.async.bulk.tensor) and the tcgen05 tensor-core/TMEM ops.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/echo.h"

namespace echo {

constexpr int kHeads = ECHO_H_INDEX;
constexpr int kDim = ECHO_D_INDEX;
constexpr int kKvElems = ECHO_KV_ELEMS;
constexpr int kKvBytes = ECHO_KV_BYTES;
constexpr int kKvChunks = kKvBytes / 16;  // 72 16-byte vectors per latent-KV row
constexpr int32_t kInf = ECHO_INF;
// a host row claimed by the selected entry f during recall: kClaim + f (< 0)
constexpr int32_t kClaim = INT32_MIN;
// GPUTokenPriority of a slot set aside for the direct-to-slot prefetch (not free,
// not evictable, no row), and of a slot the prefetch filled in this step until the
// recall gives it the step clock
constexpr int32_t kReservedPrio = -2;
constexpr int32_t kPrefetchedPrio = -3;

// wall-clock limit of every spin-wait (a second), after which the kernel flags
// ECHO_DEV_WAIT_TIMEOUT and unwinds
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void set_status(int32_t *st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

// Global reductions whose old value nobody needs: `red` lets the thread go on at once
// (an atomicAdd / atomicMin whose result is dropped may still be issued as a
// returning atomic, which waits a memory round trip).  Device memory only.
__device__ __forceinline__ void red_add(uint32_t *p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add(unsigned long long *p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_min(int32_t *p, int32_t v) {
  asm volatile("red.relaxed.gpu.global.min.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Phase tracing for development builds (-DECHO_TRACE): each translation unit keeps
// a small array of %globaltimer stamps, readable through echo_debug_trace_<unit>()
// and set to all ones by echo_debug_trace_clear_<unit>().  ECHO_TRACE_MARK is
// written by block 0, thread 0; ECHO_TRACE_FIRST keeps the earliest stamp of any
// block; ECHO_TRACE_LAST keeps the latest, stored complemented.  Product builds
// compile the marks away.
#ifdef ECHO_TRACE
static __device__ unsigned long long g_echo_trace[32];
#define ECHO_TRACE_UNIT(name)                                                                      \
  extern "C" int echo_debug_trace_##name(unsigned long long *out) {                                \
    return cudaMemcpyFromSymbol(out, echo::g_echo_trace, sizeof(echo::g_echo_trace)) == cudaSuccess \
               ? 0                                                                                 \
               : 2;                                                                                \
  }                                                                                                \
  extern "C" int echo_debug_trace_clear_##name() {                                                 \
    unsigned long long ones[32];                                                                   \
    for (int i = 0; i < 32; ++i) ones[i] = ~0ull;                                                  \
    return cudaMemcpyToSymbol(echo::g_echo_trace, ones, sizeof(ones)) == cudaSuccess ? 0 : 2;      \
  }
#define ECHO_TRACE_MARK(slot)                                                          \
  do {                                                                                 \
    if (blockIdx.x == 0 && threadIdx.x == 0) g_echo_trace[slot] = echo::globaltimer(); \
  } while (0)
#define ECHO_TRACE_FIRST(slot)                                                 \
  do {                                                                         \
    if (threadIdx.x == 0) atomicMin(&g_echo_trace[slot], echo::globaltimer()); \
  } while (0)
#define ECHO_TRACE_LAST(slot)                                                   \
  do {                                                                          \
    if (threadIdx.x == 0) atomicMin(&g_echo_trace[slot], ~echo::globaltimer()); \
  } while (0)
#define ECHO_TRACE_LAST_HERE(slot)                           \
  do {                                                       \
    atomicMin(&g_echo_trace[slot], ~echo::globaltimer());    \
  } while (0)
#define ECHO_TRACE_FIRST_HERE(slot)                          \
  do {                                                       \
    atomicMin(&g_echo_trace[slot], echo::globaltimer());     \
  } while (0)
#define ECHO_TRACE_VALUE(slot, v)                                                        \
  do {                                                                                   \
    if (blockIdx.x == 0 && threadIdx.x == 0) g_echo_trace[slot] = (unsigned long long)(v); \
  } while (0)
#define ECHO_TRACE_LAST_BLOCK(slot)                                                                   \
  do {                                                                                                \
    atomicMin(&g_echo_trace[slot], ~(((echo::globaltimer() & ((1ull << 56) - 1)) << 8) | (unsigned long long)blockIdx.x)); \
  } while (0)
#else
#define ECHO_TRACE_UNIT(name)
#define ECHO_TRACE_MARK(slot) \
  do {                        \
  } while (0)
#define ECHO_TRACE_FIRST(slot) \
  do {                         \
  } while (0)
#define ECHO_TRACE_LAST(slot) \
  do {                        \
  } while (0)
#define ECHO_TRACE_LAST_HERE(slot) \
  do {                             \
  } while (0)
#define ECHO_TRACE_FIRST_HERE(slot) \
  do {                              \
  } while (0)
#define ECHO_TRACE_VALUE(slot, v) \
  do {                            \
  } while (0)
#define ECHO_TRACE_LAST_BLOCK(slot) \
  do {                              \
  } while (0)
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

// element u of a small register array, u not known at compile time (a select
// chain keeps the array in registers instead of local memory)
template <typename T, int N>
__device__ __forceinline__ T pick_reg(const T (&a)[N], int u) {
  T x = a[0];
#pragma unroll
  for (int i = 1; i < N; ++i) x = u == i ? a[i] : x;
  return x;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the kernel before it finishes; pdl_wait() blocks
// until that kernel has completed and its memory is visible (a no-op for an
// ordinary launch).  pdl_launch_dependents() lets the next such kernel start early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Gives up (returns false) after
// kWaitLimitNs or as soon as *abort is set; a timeout sets *abort and the status
// bit so that every role of the CTA unwinds.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        set_status(status, ECHO_DEV_WAIT_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map,
                                                        uint64_t *bar, int32_t x, int32_t y,
                                                        int32_t z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 e4m3 operands, fp32 accumulator
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on `bar` once every tcgen05 op issued so far by this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Marks 32 registers as written here, so that no read of them can be scheduled above
// this point: placed right after tcgen05.wait::ld, it keeps the arithmetic on the
// loaded values behind the wait (the compiler cannot see that tcgen05.ld is
// asynchronous).
__device__ __forceinline__ void reg_fence_32(float (&v)[32]) {
  asm volatile(""
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                 "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]),
                 "+f"(v[15]), "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]),
                 "+f"(v[22]), "+f"(v[23]), "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]),
                 "+f"(v[29]), "+f"(v[30]), "+f"(v[31])
               :
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets row (lane base + i)
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand stored as rows of 128
// bytes with the 128-byte swizzle (the layout a TMA box of 128-byte rows with
// CU_TENSOR_MAP_SWIZZLE_128B produces): 8-row groups 1024 bytes apart.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4 (unused: 1)
//   bits 32-45 stride byte offset >> 4 bits 46-48 0b001 (descriptor version)
//   bits 49-51 base offset (0: 1024-byte aligned atoms)  bits 61-63 swizzle (2 = 128B)
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32, A = B = e4m3,
// both K-major, dense, shape M x N.
//   bits 4-5 D format (1 = f32), 7-9 A format (0 = e4m3), 10-12 B format,
//   15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// misc
// ---------------------------------------------------------------------------
// order-preserving map of an fp32 score onto uint32 (-0 folded onto +0): a larger
// key is a larger score
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// acc + (wx, wy) * (relu(vx), relu(vy)): two heads of the indexer's weighted ReLU sum in
// one paired fp32 FMA (each half rounds exactly as fmaf does)
__device__ __forceinline__ float2 fma_relu2(float wx, float wy, float vx, float vy, float2 acc) {
  return __ffma2_rn(make_float2(wx, wy), make_float2(fmaxf(vx, 0.f), fmaxf(vy, 0.f)), acc);
}

__device__ __forceinline__ int query_valid_len(int L, int n_q, int j) {
  int v = L - (n_q - 1 - j);
  return v < 0 ? 0 : v;
}

}  // namespace echo

// host-side error helper shared by the launchers
namespace echo_host {
void set_error(const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *what);

// Devices a process may use with the library (per-device caches are this long).
constexpr int kMaxDevices = 64;

// Raises a kernel's dynamic shared-memory limit once per device (the first call on a
// device must come before any stream capture on it), and asks for the largest
// shared-memory carveout: the kernels of a step then share one L1 / shared-memory
// split, so a kernel launched programmatically can start on an SM where the one
// before it still runs instead of waiting for the SM to drain and be reconfigured.
// Threads making their first call together may both set the attributes; the flag is
// atomic, so that is harmless.
template <typename K>
inline int smem_limit_once(std::atomic<bool> (&done)[kMaxDevices], K kernel, int bytes, const char *what) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device index %d out of range (the library serves devices 0..%d)", dev, kMaxDevices - 1);
    return ECHO_ENOTSUP;
  }
  if (done[dev].load(std::memory_order_acquire)) return 0;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_fail(e, what);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e, what);
  done[dev].store(true, std::memory_order_release);
  return 0;
}
}  // namespace echo_host
