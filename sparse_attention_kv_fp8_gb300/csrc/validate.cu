// validate.cu -- the invariants of one pool's metadata (ECHO review,
// marsggbo.github.io, "OSDI'26 | ECHO", section 5.1 metadata table: GPUTokenFree,
// GPUTokenPriority, GPUTokenToHost and HostTokenToGPU describe one bijection
// between occupied slots and resident host rows; section 5.2: a freed slot gets
// free = 1, priority = -1 and loses both map entries).
//
// The same per-slot and per-row checks run on the device (echo_pool_validate: one
// grid-stride kernel that counts violations, then one thread that compares the
// free-slot count with the pool's counter and raises ECHO_DEV_INVARIANT) and on the
// host over copies of the arrays (echo_pool_validate_host), so a test or a tool can
// look at a snapshot without a GPU.
#include <cstring>

#include "echo_common.cuh"

namespace echo {

// slot states between calls (a slot the direct-to-slot prefetch filled this step
// keeps kPrefetchedPrio until the recall that follows gives it the step clock)
__host__ __device__ inline void check_slot(int32_t s, uint8_t fr, int32_t pr, int32_t th, const int32_t *h2g,
                                           int32_t n_h, int32_t *rep) {
  if (fr == 1) {
    ++rep[ECHO_VAL_FREE];
    if (pr != -1 || th != kInf) ++rep[ECHO_VAL_SLOT_STATE];
    return;
  }
  if (fr != 0) {
    ++rep[ECHO_VAL_SLOT_STATE];
    return;
  }
  if (pr == kReservedPrio) {
    ++rep[ECHO_VAL_RESERVED];
    rep[ECHO_VAL_BALANCE] = static_cast<int32_t>(static_cast<uint32_t>(rep[ECHO_VAL_BALANCE]) + static_cast<uint32_t>(s));
    if (th != kInf) ++rep[ECHO_VAL_SLOT_STATE];
    return;
  }
  ++rep[ECHO_VAL_OCCUPIED];
  if (pr < 0 && pr != kPrefetchedPrio) ++rep[ECHO_VAL_SLOT_STATE];
  if (th < 0 || th >= n_h) {
    ++rep[ECHO_VAL_SLOT_STATE];
  } else if (h2g[th] != s) {
    ++rep[ECHO_VAL_SLOT_MAP];
  }
}

__host__ __device__ inline void check_row(int32_t h, int32_t v, const int32_t *to_host, int32_t n_g, int32_t *rep) {
  if (v == kInf) return;
  ++rep[ECHO_VAL_RESIDENT];
  if (v < 0 || v >= n_g || to_host[v] != h) ++rep[ECHO_VAL_ROW_MAP];
}

__host__ __device__ inline void check_reserve_entry(int32_t s, const int32_t *prio, int32_t n_g, int32_t *rep) {
  if (s < 0 || s >= n_g || prio[s] != kReservedPrio) ++rep[ECHO_VAL_RESERVE];
  rep[ECHO_VAL_BALANCE] = static_cast<int32_t>(static_cast<uint32_t>(rep[ECHO_VAL_BALANCE]) - static_cast<uint32_t>(s));
}

// the comparisons that need every count: free slots against the pool's counter,
// reserved slots against the reserve's length
__host__ __device__ inline void check_totals(int32_t n_free_counter, int32_t res_len, bool with_reserve,
                                             int32_t *rep) {
  if (rep[ECHO_VAL_FREE] != n_free_counter) ++rep[ECHO_VAL_COUNTER];
  if (with_reserve && (rep[ECHO_VAL_RESERVED] != res_len || rep[ECHO_VAL_BALANCE] != 0)) ++rep[ECHO_VAL_RESERVE];
}

__host__ __device__ inline bool any_violation(const int32_t *rep) {
  return rep[ECHO_VAL_SLOT_STATE] | rep[ECHO_VAL_SLOT_MAP] | rep[ECHO_VAL_ROW_MAP] | rep[ECHO_VAL_COUNTER] |
         rep[ECHO_VAL_RESERVE];
}

constexpr int kValThreads = 256;

__global__ void __launch_bounds__(kValThreads) validate_kernel(const uint8_t *free_, const int32_t *prio,
                                                               const int32_t *to_host, const int32_t *h2g,
                                                               int32_t n_g, int32_t n_h, const int32_t *reserve,
                                                               const int32_t *reserve_ctl, int32_t res_cap,
                                                               int32_t *report) {
  __shared__ int32_t blk[ECHO_VAL_COUNT];
  if (threadIdx.x < ECHO_VAL_COUNT) blk[threadIdx.x] = 0;
  __syncthreads();
  int32_t rep[ECHO_VAL_COUNT];
#pragma unroll
  for (int i = 0; i < ECHO_VAL_COUNT; ++i) rep[i] = 0;
  const int tid = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
  for (int s = tid; s < n_g; s += nt) check_slot(s, free_[s], prio[s], to_host[s], h2g, n_h, rep);
  for (int h = tid; h < n_h; h += nt) check_row(h, h2g[h], to_host, n_g, rep);
  if (reserve) {
    // the reserve array holds res_cap entries: a longer recorded length is itself a
    // violation (found by the finishing kernel) and is not followed past the array
    const int32_t len = min(reserve_ctl[1], res_cap);
    for (int i = tid; i < len; i += nt) check_reserve_entry(reserve[i], prio, n_g, rep);
  }
  // counts and the (mod 2^32) balance add the same way as unsigned words
#pragma unroll
  for (int i = 0; i < ECHO_VAL_COUNT; ++i)
    if (rep[i]) atomicAdd(reinterpret_cast<unsigned *>(&blk[i]), static_cast<unsigned>(rep[i]));
  __syncthreads();
  if (threadIdx.x < ECHO_VAL_COUNT && blk[threadIdx.x])
    atomicAdd(reinterpret_cast<unsigned *>(report + threadIdx.x), static_cast<unsigned>(blk[threadIdx.x]));
}

__global__ void validate_finish_kernel(const int32_t *counters, const int32_t *reserve_ctl, int32_t res_cap,
                                       int32_t *report, int32_t *status) {
  const int32_t len = reserve_ctl ? reserve_ctl[1] : 0;
  if (reserve_ctl && (len < 0 || len > res_cap)) ++report[ECHO_VAL_RESERVE];
  check_totals(counters[0], len, reserve_ctl != nullptr, report);
  if (any_violation(report)) set_status(status, ECHO_DEV_INVARIANT);
}

}  // namespace echo

namespace echo_host {

int sm_count();

int launch_validate(const echo_pool *p, const echo_stage *stage, int32_t *report, int32_t *status,
                    cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(report, 0, ECHO_VAL_COUNT * sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "validate: clearing the report");
  const long long n = p->n_h > p->n_g ? p->n_h : p->n_g;
  long long grid = (n + echo::kValThreads - 1) / echo::kValThreads;
  const long long cap = static_cast<long long>(sm_count()) * 4;
  grid = grid > cap ? cap : (grid < 1 ? 1 : grid);
  const int32_t *reserve = stage ? stage->reserve : nullptr;
  const int32_t *reserve_ctl = stage ? stage->reserve_ctl : nullptr;
  const int32_t res_cap = stage ? stage->reserve_cap : 0;
  echo::validate_kernel<<<static_cast<int>(grid), echo::kValThreads, 0, s>>>(
      p->gpu_token_free, p->gpu_token_priority, p->gpu_token_to_host, p->host_token_to_gpu, p->n_g, p->n_h, reserve,
      reserve_ctl, res_cap, report);
  echo::validate_finish_kernel<<<1, 1, 0, s>>>(p->counters, reserve_ctl, res_cap, report, status);
  e = cudaGetLastError();
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "validate launch");
}

int validate_host(const echo_pool *p, const int32_t *reserve, int32_t reserve_len, int32_t *report) {
  std::memset(report, 0, ECHO_VAL_COUNT * sizeof(int32_t));
  for (int32_t s = 0; s < p->n_g; ++s)
    echo::check_slot(s, p->gpu_token_free[s], p->gpu_token_priority[s], p->gpu_token_to_host[s],
                     p->host_token_to_gpu, p->n_h, report);
  for (int32_t h = 0; h < p->n_h; ++h) echo::check_row(h, p->host_token_to_gpu[h], p->gpu_token_to_host, p->n_g, report);
  if (reserve)
    for (int32_t i = 0; i < reserve_len && i < p->n_g; ++i)
      echo::check_reserve_entry(reserve[i], p->gpu_token_priority, p->n_g, report);
  echo::check_totals(p->counters[0], reserve_len, reserve != nullptr, report);
  return echo::any_violation(report) ? ECHO_DEV_INVARIANT : 0;
}

}  // namespace echo_host
