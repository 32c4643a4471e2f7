// api.cu -- the extern "C" entry points declared in include/echo.h: argument
// validation on the host, then kernel launches on the caller's stream.  Nothing
// here allocates, synchronises or reads device memory.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "cache_common.cuh"

namespace echo_host {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

int cuda_fail(cudaError_t e, const char *what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return ECHO_ECUDA;
}

// launchers (indexer.cu, topk.cu, cache_mgr.cu)
int launch_indexer(const echo_indexer_args *a, cudaStream_t stream);
int launch_indexer(const echo_indexer_args *a, cudaStream_t stream, uint32_t *sel_hist, const int4 *sel_hint);
echo::Workspace workspace_view(const echo_workspace *w);
int launch_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                float *kth, cudaStream_t stream);
size_t workspace_bytes(int32_t n_g, int32_t max_rows);
int launch_workspace_init(const echo_workspace *w, cudaStream_t s);
int launch_pool_init(const echo_pool *p, cudaStream_t s);
int launch_pool_alloc(const echo_pool *pool, const echo_workspace *ws, const int32_t *host_idx, const int32_t *n_dev,
                      int32_t max_n, int32_t clock, const int32_t *clock_dev, int32_t *out_slots, int32_t *status,
                      cudaStream_t s);
int launch_pool_evict(const echo_pool *pool, const echo_workspace *ws, const int32_t *n_needed_dev, int32_t clock,
                      const int32_t *clock_dev, int32_t *status, cudaStream_t s);
int launch_recall(const echo_pool *pool, const echo_workspace *ws, const int32_t *sel, const int32_t *req_to_host,
                  const int32_t *ctx_len, int B, int n_q, int k, int L_max, const echo_stage *stage, int32_t clock,
                  const int32_t *clock_dev, int32_t *out_slot, echo_stats *stats, int32_t *status, cudaStream_t s,
                  float *ema_s_hat, const float *ema_kth, int ema_n, float ema_alpha, int32_t *clock_advance,
                  int claimed);
int launch_topk_claim(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max, int k, int32_t *sel,
                      float *kth, const echo_pool *pool, const echo_workspace *ws, const int32_t *req_to_host,
                      int32_t clock, const int32_t *clock_dev, int32_t *status, cudaStream_t stream);
int launch_wait_probe(int which, int32_t *status, cudaStream_t s);
int launch_append(const echo_pool *pool, const echo_workspace *ws, uint8_t *k_index, int32_t *ctx_len,
                  const int32_t *req_to_host, int B, int L_max, const uint16_t *new_kv, const uint8_t *new_k_index,
                  int32_t clock, const int32_t *clock_dev, echo_stats *stats, int32_t *status, cudaStream_t s);
int launch_ema(float *s_hat, const float *kth, int n, int stride, float alpha, cudaStream_t s);
int launch_prefill_indexer(const echo_prefill_args *a, cudaStream_t stream);
size_t mla_workspace_bytes(int32_t B, int32_t n_q, int32_t k);
int launch_sparse_mla(const echo_mla_args *a, cudaStream_t stream);
int noalloc_workspace(int32_t n_g, int32_t rows, cudaStream_t stream, echo_workspace *out);
int launch_validate(const echo_pool *p, const echo_stage *stage, int32_t *report, int32_t *status, cudaStream_t s);
int validate_host(const echo_pool *p, const int32_t *reserve, int32_t reserve_len, int32_t *report);

}  // namespace echo_host

using namespace echo_host;

#define REQUIRE(cond, ...)             \
  do {                                 \
    if (!(cond)) {                     \
      set_error(__VA_ARGS__);          \
      return ECHO_EINVAL;              \
    }                                  \
  } while (0)

#define TRY(x)                  \
  do {                          \
    int _r = (x);               \
    if (_r != ECHO_OK) return _r; \
  } while (0)

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A pointer the kernels may dereference: device memory, managed memory, or
// pinned host memory mapped at the same address.  Checked once per pointer (the
// answer is cached) so that later calls stay capturable.
static int check_device_accessible(const void *p, const char *name) {
  static std::mutex mu;
  static const void *seen[64];
  static int n_seen = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_seen; ++i)
      if (seen[i] == p) return ECHO_OK;
  }
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    set_error("%s: not a CUDA-visible pointer (%s)", name, cudaGetErrorString(e));
    return ECHO_EINVAL;
  }
  bool ok = at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged ||
            (at.type == cudaMemoryTypeHost && at.devicePointer == p);
  if (!ok) {
    set_error("%s: must be device memory or pinned host memory mapped at the same address", name);
    return ECHO_EINVAL;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (n_seen < 64) seen[n_seen++] = p;
  return ECHO_OK;
}

static int check_pool(const echo_pool *p) {
  REQUIRE(p, "pool is NULL");
  REQUIRE(p->n_g > 0 && p->n_h > 0, "pool sizes must be positive (n_g=%d, n_h=%d)", p->n_g, p->n_h);
  REQUIRE(p->row_elems >= 0 && p->row_elems <= 65536 && p->row_elems % 8 == 0,
          "row_elems must be 0 (576) or a multiple of 8 up to 65536 (got %d)", p->row_elems);
  REQUIRE(p->gpu_token_free && p->gpu_token_priority && p->gpu_indices_buffer && p->gpu_token_to_host &&
              p->host_token_to_gpu && p->counters,
          "pool metadata pointer is NULL");
  REQUIRE(p->gpu_kv && p->host_kv, "pool KV pointer is NULL");
  REQUIRE(aligned(p->gpu_kv, 16) && aligned(p->host_kv, 16), "pool KV pools must be 16-byte aligned");
  return check_device_accessible(p->host_kv, "pool.host_kv");
}

// The calls that prefetch copy MLA latent rows (576 bf16) by a fixed layout.
static int check_latent_rows(const echo_pool *p, const char *what) {
  REQUIRE(p->row_elems == 0 || p->row_elems == ECHO_KV_ELEMS, "%s needs a pool of %d-element rows (row_elems %d)",
          what, ECHO_KV_ELEMS, p->row_elems);
  return ECHO_OK;
}

static int check_ws(const echo_workspace *w, const echo_pool *p, long long rows) {
  REQUIRE(w && w->base, "workspace is NULL");
  REQUIRE(aligned(w->base, 256), "workspace base must be 256-byte aligned");
  REQUIRE(w->n_g == p->n_g, "workspace was sized for n_g=%d, pool has %d", w->n_g, p->n_g);
  REQUIRE(rows <= w->max_rows, "call needs %lld workspace rows, workspace has %d", rows, w->max_rows);
  REQUIRE(w->bytes >= workspace_bytes(w->n_g, w->max_rows), "workspace smaller than echo_workspace_bytes()");
  return ECHO_OK;
}

static int check_stage(const echo_stage *st, const echo_pool *pool) {
  REQUIRE((st->flags & ~ECHO_PREFETCH_WHILE_SCORING) == 0, "unknown stage flags 0x%x", st->flags);
  if (st->reserve) {  // direct to slot
    REQUIRE(st->reserve_ctl, "direct-to-slot stage without reserve_ctl");
    REQUIRE(st->reserve_cap >= 0 && st->reserve_cap <= pool->n_g,
            "reserve_cap must be in [0, n_g] (got %d, n_g %d)", st->reserve_cap, pool->n_g);
    return ECHO_OK;
  }
  REQUIRE(st->rows && st->host_row && st->count, "stage pointer is NULL");
  REQUIRE(aligned(st->rows, 16), "stage rows must be 16-byte aligned");
  REQUIRE(st->stride > 0 && st->cap_div > 0, "stage stride and cap_div must be positive");
  return ECHO_OK;
}

extern "C" {

const char *echo_last_error_string(void) { return g_err; }

int echo_selftest_wait_timeout(int32_t which, int32_t *dev_status, void *stream) {
  REQUIRE(which == 0 || which == 1, "which must be 0 (mbarrier wait) or 1 (grid barrier)");
  REQUIRE(dev_status, "dev_status is NULL");
  return launch_wait_probe(which, dev_status, static_cast<cudaStream_t>(stream));
}

int32_t echo_version(void) { return (1 << 16) | 5; }

int64_t echo_metadata_bytes(int64_t n_h, int64_t n_g) {
  return static_cast<int64_t>(sizeof(int32_t)) * n_h +
         static_cast<int64_t>(sizeof(uint8_t) + 3 * sizeof(int32_t)) * n_g;
}

int echo_pool_validate(const echo_pool *pool, const echo_stage *stage, int32_t *report, int32_t *dev_status,
                       void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(report && dev_status, "validate needs report and dev_status");
  REQUIRE(!stage || (stage->reserve && stage->reserve_ctl), "validate's stage must be a direct-to-slot stage");
  return launch_validate(pool, stage, report, dev_status, static_cast<cudaStream_t>(stream));
}

int echo_pool_validate_host(const echo_pool *p, const int32_t *reserve, int32_t reserve_len, int32_t *report) {
  g_err[0] = 0;
  if (!p || !report || p->n_g <= 0 || p->n_h <= 0 || !p->gpu_token_free || !p->gpu_token_priority ||
      !p->gpu_token_to_host || !p->host_token_to_gpu || !p->counters || reserve_len < 0 ||
      (reserve_len > 0 && !reserve)) {
    set_error("echo_pool_validate_host: bad arguments");
    return -ECHO_EINVAL;
  }
  return validate_host(p, reserve, reserve_len, report);
}

// the indexer's checks and launch; the decode step also hands it the workspace's
// selection histograms (sel_hist / sel_hint, null for the public call)
static int indexer_call(const echo_indexer_args *a, void *stream, uint32_t *sel_hist, const int4 *sel_hint) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->q && a->w && a->k_index && a->ctx_len && a->scores, "indexer pointer is NULL");
  REQUIRE(a->B >= 0 && a->L_max >= 0, "negative size");
  REQUIRE(a->n_q == 1 || a->n_q == 2, "n_q must be 1 or 2 (got %d)", a->n_q);
  REQUIRE(aligned(a->q, 16) && aligned(a->k_index, 16), "q and k_index must be 16-byte aligned");
  REQUIRE(static_cast<long long>(a->B) * a->L_max <= (1ll << 31) - 1, "B * L_max too large");
  REQUIRE(static_cast<long long>(a->B) * a->n_q * echo::kHeads <= (1ll << 31) - 1, "B too large");
  if (a->s_hat) {
    REQUIRE(a->req_to_host && a->pool && a->stage, "prefetch needs req_to_host, pool and stage");
    TRY(check_pool(a->pool));
    TRY(check_latent_rows(a->pool, "the indexer's prefetch"));
    TRY(check_stage(a->stage, a->pool));
    REQUIRE(a->stage->reserve || static_cast<long long>(a->B) * a->stage->stride <= (1ll << 31) - 1,
            "stage too large");
  }
  if (a->B == 0 || a->L_max == 0) return ECHO_OK;
  return launch_indexer(a, static_cast<cudaStream_t>(stream), sel_hist, sel_hint);
}

extern "C" int echo_indexer_score(const echo_indexer_args *a, void *stream) {
  g_err[0] = 0;
  return indexer_call(a, stream, nullptr, nullptr);
}

int echo_select_topk(const float *scores, const int32_t *ctx_len, int32_t B, int32_t n_q, int32_t L_max, int32_t k,
                     int32_t *sel, float *kth, void *stream) {
  g_err[0] = 0;
  REQUIRE(scores && ctx_len && sel && kth, "top-k pointer is NULL");
  REQUIRE(B >= 0 && L_max >= 0, "negative size");
  REQUIRE(n_q >= 1 && n_q <= 65536, "n_q must be in [1, 65536] (got %d)", n_q);
  REQUIRE(k >= 1 && k <= 8192, "k must be in [1, 8192] (got %d)", k);
  REQUIRE(static_cast<long long>(B) * n_q * 8 <= (1ll << 31) - 1, "B too large");
  if (B == 0) return ECHO_OK;
  return launch_topk(scores, ctx_len, B, n_q, L_max, k, sel, kth, static_cast<cudaStream_t>(stream));
}

int echo_workspace_bytes(int32_t n_g, int32_t max_rows, size_t *bytes) {
  g_err[0] = 0;
  REQUIRE(bytes, "bytes is NULL");
  REQUIRE(n_g > 0 && max_rows >= 0, "bad workspace sizes");
  *bytes = workspace_bytes(n_g, max_rows);
  return ECHO_OK;
}

int echo_workspace_init(const echo_workspace *ws, void *stream) {
  g_err[0] = 0;
  REQUIRE(ws && ws->base, "workspace is NULL");
  REQUIRE(aligned(ws->base, 256), "workspace base must be 256-byte aligned");
  REQUIRE(ws->n_g > 0 && ws->max_rows >= 0, "bad workspace sizes");
  REQUIRE(ws->bytes >= workspace_bytes(ws->n_g, ws->max_rows), "workspace smaller than echo_workspace_bytes()");
  return launch_workspace_init(ws, static_cast<cudaStream_t>(stream));
}

int echo_pool_init(const echo_pool *pool, void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  return launch_pool_init(pool, static_cast<cudaStream_t>(stream));
}

int echo_pool_alloc(const echo_pool *pool, const echo_workspace *ws, const int32_t *host_idx, const int32_t *n_dev,
                    int32_t max_n, int32_t clock, const int32_t *clock_dev, int32_t *out_slots, int32_t *dev_status,
                    void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(max_n >= 0, "max_n must be >= 0");
  REQUIRE(n_dev && (max_n == 0 || (host_idx && out_slots)), "allocate pointer is NULL");
  REQUIRE(clock >= 0 || clock_dev, "clock must be >= 0");
  TRY(check_ws(ws, pool, max_n));
  return launch_pool_alloc(pool, ws, host_idx, n_dev, max_n, clock, clock_dev, out_slots, dev_status,
                           static_cast<cudaStream_t>(stream));
}

int echo_pool_evict(const echo_pool *pool, const echo_workspace *ws, const int32_t *n_needed_dev, int32_t clock,
                    const int32_t *clock_dev, int32_t *dev_status, void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(n_needed_dev, "n_needed_dev is NULL");
  REQUIRE(clock >= 0 || clock_dev, "clock must be >= 0");
  TRY(check_ws(ws, pool, 0));
  return launch_pool_evict(pool, ws, n_needed_dev, clock, clock_dev, dev_status, static_cast<cudaStream_t>(stream));
}

int echo_prefetch_recall(const echo_pool *pool, const echo_workspace *ws, const int32_t *sel,
                         const int32_t *req_to_host, const int32_t *ctx_len, int32_t B, int32_t n_q, int32_t k,
                         int32_t L_max, const echo_stage *stage, int32_t clock, const int32_t *clock_dev,
                         int32_t *out_slot, echo_stats *stats, int32_t *dev_status, void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(B >= 0 && L_max >= 0 && k >= 1, "bad sizes");
  REQUIRE(n_q >= 1 && n_q <= 65536, "n_q must be in [1, 65536]");
  REQUIRE(B == 0 || (sel && req_to_host && out_slot && ctx_len), "recall pointer is NULL");
  REQUIRE(clock >= 0 || clock_dev, "clock must be >= 0");
  const long long F = static_cast<long long>(B) * n_q * k;
  REQUIRE(F <= (1ll << 30), "B * n_q * k too large");
  TRY(check_ws(ws, pool, F));
  if (stage) {
    TRY(check_latent_rows(pool, "a recall with a stage"));
    TRY(check_stage(stage, pool));
  }
  return launch_recall(pool, ws, sel, req_to_host, ctx_len, B, n_q, k, L_max, stage, clock, clock_dev, out_slot, stats,
                       dev_status, static_cast<cudaStream_t>(stream), nullptr, nullptr, 0, 0.f, nullptr, 0);
}

int echo_prefetch_recall_noalloc(const echo_pool *pool, const int32_t *sel, const int32_t *req_to_host,
                                 const int32_t *ctx_len, int32_t B, int32_t n_q, int32_t k, int32_t L_max,
                                 const echo_stage *stage, int32_t clock, const int32_t *clock_dev, int32_t *out_slot,
                                 echo_stats *stats, int32_t *dev_status, void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(B >= 0 && L_max >= 0 && k >= 1, "bad sizes");
  REQUIRE(n_q >= 1 && n_q <= 65536, "n_q must be in [1, 65536]");
  REQUIRE(B == 0 || (sel && req_to_host && out_slot && ctx_len), "recall pointer is NULL");
  REQUIRE(clock >= 0 || clock_dev, "clock must be >= 0");
  const long long F = static_cast<long long>(B) * n_q * k;
  REQUIRE(F <= (1ll << 30), "B * n_q * k too large");
  if (stage) {
    TRY(check_latent_rows(pool, "a recall with a stage"));
    TRY(check_stage(stage, pool));
  }
  echo_workspace ws;
  TRY(noalloc_workspace(pool->n_g, static_cast<int32_t>(F), static_cast<cudaStream_t>(stream), &ws));
  // the array keeps whatever the last call left: lay it out for this call and reset it
  TRY(launch_workspace_init(&ws, static_cast<cudaStream_t>(stream)));
  return launch_recall(pool, &ws, sel, req_to_host, ctx_len, B, n_q, k, L_max, stage, clock, clock_dev, out_slot,
                       stats, dev_status, static_cast<cudaStream_t>(stream), nullptr, nullptr, 0, 0.f, nullptr, 0);
}

int echo_append(const echo_pool *pool, const echo_workspace *ws, uint8_t *k_index, int32_t *ctx_len,
                const int32_t *req_to_host, int32_t B, int32_t L_max, const uint16_t *new_kv,
                const uint8_t *new_k_index, int32_t clock, const int32_t *clock_dev, echo_stats *stats,
                int32_t *dev_status, void *stream) {
  g_err[0] = 0;
  TRY(check_pool(pool));
  REQUIRE(B >= 0 && L_max >= 0, "bad sizes");
  REQUIRE(B == 0 || (k_index && ctx_len && req_to_host && new_kv && new_k_index), "append pointer is NULL");
  REQUIRE(aligned(new_kv, 16) && aligned(new_k_index, 16) && aligned(k_index, 16), "append buffers must be 16-byte aligned");
  REQUIRE(clock >= 0 || clock_dev, "clock must be >= 0");
  TRY(check_ws(ws, pool, B));
  return launch_append(pool, ws, k_index, ctx_len, req_to_host, B, L_max, new_kv, new_k_index, clock, clock_dev, stats,
                       dev_status, static_cast<cudaStream_t>(stream));
}

int echo_ema_update(float *s_hat, const float *kth, int32_t n, float alpha, void *stream) {
  g_err[0] = 0;
  REQUIRE(n >= 0, "n must be >= 0");
  REQUIRE(n == 0 || (s_hat && kth), "EMA pointer is NULL");
  REQUIRE(alpha >= 0.f && alpha <= 1.f, "alpha must be in [0, 1]");
  if (n == 0) return ECHO_OK;
  return launch_ema(s_hat, kth, n, 1, alpha, static_cast<cudaStream_t>(stream));
}

int echo_ema_update_strided(float *s_hat, const float *kth, int32_t n, int32_t kth_stride, float alpha,
                            void *stream) {
  g_err[0] = 0;
  REQUIRE(n >= 0, "n must be >= 0");
  REQUIRE(kth_stride >= 1, "kth_stride must be >= 1");
  REQUIRE(n == 0 || (s_hat && kth), "EMA pointer is NULL");
  REQUIRE(alpha >= 0.f && alpha <= 1.f, "alpha must be in [0, 1]");
  REQUIRE(static_cast<long long>(n) * kth_stride <= (1ll << 31) - 1, "n * kth_stride too large");
  if (n == 0) return ECHO_OK;
  return launch_ema(s_hat, kth, n, kth_stride, alpha, static_cast<cudaStream_t>(stream));
}

int echo_mla_workspace_bytes(int32_t B, int32_t n_q, int32_t k, size_t *bytes) {
  g_err[0] = 0;
  REQUIRE(bytes, "bytes is NULL");
  REQUIRE(B >= 0 && n_q >= 1 && n_q <= 65536 && k >= 1 && k <= 8192, "bad sizes (B %d, n_q %d, k %d)", B, n_q, k);
  *bytes = mla_workspace_bytes(B, n_q, k);
  return ECHO_OK;
}

int echo_sparse_mla_decode(const echo_mla_args *a, void *stream) {
  g_err[0] = 0;
  REQUIRE(a, "args is NULL");
  REQUIRE(a->B >= 0 && a->n_q >= 1 && a->n_q <= 65536, "bad sizes (B %d, n_q %d)", a->B, a->n_q);
  REQUIRE(a->k >= 1 && a->k <= 8192, "k must be in [1, 8192] (got %d)", a->k);
  REQUIRE(a->n_g >= 1, "n_g must be >= 1");
  if (a->B == 0) return ECHO_OK;
  REQUIRE(a->q && a->gpu_kv && a->out_slot && a->out && a->lse && a->workspace, "MLA pointer is NULL");
  REQUIRE(aligned(a->q, 16) && aligned(a->gpu_kv, 16), "q and gpu_kv must be 16-byte aligned");
  REQUIRE(aligned(a->out, 16) && aligned(a->workspace, 256), "out must be 16-byte and workspace 256-byte aligned");
  REQUIRE(static_cast<long long>(a->B) * a->n_q * 128 <= (1ll << 31) - 1, "B * n_q too large");
  REQUIRE(std::isfinite(a->scale), "scale must be finite");
  REQUIRE(a->workspace_bytes >= mla_workspace_bytes(a->B, a->n_q, a->k), "workspace smaller than "
          "echo_mla_workspace_bytes()");
  return launch_sparse_mla(a, static_cast<cudaStream_t>(stream));
}

int echo_prefill_indexer_score(const echo_prefill_args *a, void *stream) {
  g_err[0] = 0;
  REQUIRE(a, "args is NULL");
  REQUIRE(a->q && a->w && a->k_index && a->ctx_len && a->scores, "prefill indexer pointer is NULL");
  REQUIRE(a->B >= 0 && a->L_max >= 0, "negative size");
  REQUIRE(a->C >= 1 && a->C <= 65536, "C must be in [1, 65536] (got %d)", a->C);
  REQUIRE(aligned(a->q, 16) && aligned(a->k_index, 16) && aligned(a->w, 16),
          "q, w and k_index must be 16-byte aligned");
  REQUIRE(static_cast<long long>(a->B) * a->L_max <= (1ll << 31) - 1, "B * L_max too large");
  REQUIRE(static_cast<long long>(a->B) * a->C * echo::kHeads <= (1ll << 31) - 1, "B * C too large");
  REQUIRE(static_cast<long long>(a->B) * a->C * a->L_max <= (1ll << 40), "scores too large");
  if (a->s_shift) {
    REQUIRE(a->k >= 1, "k must be >= 1 with s_shift");
    if (a->stage) {
      REQUIRE(a->req_to_host && a->pool, "prefetch needs req_to_host and pool");
      TRY(check_pool(a->pool));
      TRY(check_latent_rows(a->pool, "the prefill prefetch"));
      TRY(check_stage(a->stage, a->pool));
    }
  }
  if (a->B == 0 || a->L_max == 0) return ECHO_OK;
  return launch_prefill_indexer(a, static_cast<cudaStream_t>(stream));
}

// the decode step's argument checks (everything, before anything is enqueued)
static int step_check(const echo_step_args *a) {
  REQUIRE(a, "args is NULL");
  REQUIRE(a->pool && a->ws, "step needs pool and workspace");
  REQUIRE(a->q && a->w && a->k_index && a->ctx_len && a->req_to_host && a->scores && a->sel && a->kth &&
              a->out_slot,
          "step pointer is NULL");
  REQUIRE(a->clock >= 0 || a->clock_dev, "clock must be >= 0");
  const bool prefetch = a->s_hat && a->stage;
  TRY(check_pool(a->pool));
  TRY(check_latent_rows(a->pool, "the decode step"));
  REQUIRE(a->B >= 0 && a->L_max >= 0, "negative size");
  REQUIRE(a->n_q == 1 || a->n_q == 2, "n_q must be 1 or 2 (got %d)", a->n_q);
  REQUIRE(a->k >= 1 && a->k <= 8192, "k must be in [1, 8192] (got %d)", a->k);
  REQUIRE(aligned(a->q, 16) && aligned(a->k_index, 16), "q and k_index must be 16-byte aligned");
  REQUIRE(static_cast<long long>(a->B) * a->L_max <= (1ll << 31) - 1, "B * L_max too large");
  const long long F = static_cast<long long>(a->B) * a->n_q * a->k;
  REQUIRE(F <= (1ll << 30), "B * n_q * k too large");
  TRY(check_ws(a->ws, a->pool, F > a->B ? F : a->B));
  REQUIRE(a->alpha >= 0.f && a->alpha <= 1.f, "alpha must be in [0, 1]");
  if (prefetch) TRY(check_stage(a->stage, a->pool));
  if (a->new_kv) {
    REQUIRE(a->new_k_index, "new_kv given without new_k_index");
    REQUIRE(aligned(a->new_kv, 16) && aligned(a->new_k_index, 16), "append buffers must be 16-byte aligned");
  }
  return ECHO_OK;
}

// the decode step's launches (arguments already checked)
static int step_enqueue(const echo_step_args *a, cudaStream_t s) {
  void *stream = s;
  const bool prefetch = a->s_hat && a->stage;
  cudaEvent_t *ev = reinterpret_cast<cudaEvent_t *>(a->stage_events);
  // under stream capture the records become external event nodes of the graph (so
  // that they still time each replay); outside capture they are plain records (the
  // external flag is refused there)
  unsigned int ev_flags = cudaEventRecordDefault;
  if (ev) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return cuda_fail(e, "stream capture status");
    if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
  }
  auto mark = [&](int i) -> int {
    if (!ev || !ev[i]) return ECHO_OK;
    cudaError_t e = cudaEventRecordWithFlags(ev[i], s, ev_flags);
    return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "stage event");
  };
  TRY(mark(ECHO_STAGE_APPEND));
  if (a->new_kv) {
    TRY(echo_append(a->pool, a->ws, a->k_index, a->ctx_len, a->req_to_host, a->B, a->L_max, a->new_kv,
                    a->new_k_index, a->clock, a->clock_dev, a->stats, a->dev_status, stream));
  }
  TRY(mark(ECHO_STAGE_INDEXER));
  echo_indexer_args ia{};
  ia.q = a->q;
  ia.w = a->w;
  ia.k_index = a->k_index;
  ia.ctx_len = a->ctx_len;
  ia.B = a->B;
  ia.n_q = a->n_q;
  ia.L_max = a->L_max;
  ia.scores = a->scores;
  ia.dev_status = a->dev_status;
  if (prefetch) {
    ia.s_hat = a->s_hat;
    ia.req_to_host = a->req_to_host;
    ia.pool = a->pool;
    ia.stage = a->stage;
  }
  {
    // the indexer also fills the score histograms the top-k starts from
    const echo::Workspace wv = workspace_view(a->ws);
    TRY(indexer_call(&ia, stream, wv.sel_hist, wv.sel_hint));
  }
  TRY(mark(ECHO_STAGE_TOPK));
  // the top-k kernel also makes the recall's claims for the entries it selects
  TRY(launch_topk_claim(a->scores, a->ctx_len, a->B, a->n_q, a->L_max, a->k, a->sel, a->kth, a->pool, a->ws,
                        a->req_to_host, a->clock, a->clock_dev, a->dev_status, s));
  TRY(mark(ECHO_STAGE_RECALL));
  {
    // the recall kernel also updates the EMA and advances the device clock
    TRY(launch_recall(a->pool, a->ws, a->sel, a->req_to_host, a->ctx_len, a->B, a->n_q, a->k, a->L_max,
                      prefetch ? a->stage : nullptr, a->clock, a->clock_dev, a->out_slot, a->stats, a->dev_status, s,
                      a->s_hat, a->kth, a->B * a->n_q, a->alpha,
                      (a->clock_dev && a->advance_clock) ? a->clock_dev : nullptr, 1));
  }
  TRY(mark(ECHO_STAGE_EMA));  // the EMA ran inside the recall: this stage is empty
  TRY(mark(ECHO_NUM_STAGES));
  return ECHO_OK;
}

int echo_decode_step(const echo_step_args *a, void *stream) {
  g_err[0] = 0;
  // everything is checked before the first launch, so a rejected step enqueues nothing
  TRY(step_check(a));
  return step_enqueue(a, static_cast<cudaStream_t>(stream));
}

// The step's inputs from host memory: q (B * n_q * 64 * 128 bytes) into a->q and w
// (B * n_q * 64 floats) into a->w, in one copy when both sides hold w right after q.
static int copy_step_inputs(const echo_step_args *a, const void *q_host, const float *w_host, cudaStream_t s) {
  const size_t qb = static_cast<size_t>(a->B) * a->n_q * 64 * 128;
  const size_t wb = static_cast<size_t>(a->B) * a->n_q * 64 * sizeof(float);
  if (qb == 0) return ECHO_OK;
  const uint8_t *qh = static_cast<const uint8_t *>(q_host);
  const uint8_t *qd = a->q;
  cudaError_t e;
  if (reinterpret_cast<const uint8_t *>(w_host) == qh + qb && reinterpret_cast<const uint8_t *>(a->w) == qd + qb) {
    e = cudaMemcpyAsync(const_cast<uint8_t *>(qd), qh, qb + wb, cudaMemcpyHostToDevice, s);
  } else {
    e = cudaMemcpyAsync(const_cast<uint8_t *>(qd), qh, qb, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(const_cast<float *>(a->w), w_host, wb, cudaMemcpyHostToDevice, s);
  }
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "input copy");
}

static int wait_stream(cudaStream_t s) {
  const cudaError_t e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? ECHO_OK : cuda_fail(e, "stream synchronisation");
}

int echo_decode_step_host(const echo_step_args *a, const void *q_host, const float *w_host, void *stream,
                          int32_t wait) {
  g_err[0] = 0;
  REQUIRE(q_host && w_host, "q_host and w_host are required");
  TRY(step_check(a));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TRY(copy_step_inputs(a, q_host, w_host, s));
  TRY(step_enqueue(a, s));
  return wait ? wait_stream(s) : ECHO_OK;
}

}  // extern "C"

// A decode step captured once into a CUDA graph by the library (its own capture
// stream), replayed by echo_step_graph_launch.
struct echo_step_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  echo_step_args args;
};

extern "C" {

int echo_step_graph_create(const echo_step_args *a, echo_step_graph **out) {
  g_err[0] = 0;
  REQUIRE(out, "out is NULL");
  *out = nullptr;
  REQUIRE(a, "args is NULL");
  REQUIRE(a->clock_dev, "a step graph needs the device clock (clock_dev) so that each launch is the next step");
  REQUIRE(!a->stage_events, "a step graph takes no stage events");
  TRY(step_check(a));
  cudaStream_t cs = nullptr;
  cudaError_t e = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking);
  if (e != cudaSuccess) return cuda_fail(e, "capture stream");
  // relaxed: the first launches of a process set kernel attributes inside the capture
  e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) {
    cudaStreamDestroy(cs);
    return cuda_fail(e, "begin capture");
  }
  const int rc = step_enqueue(a, cs);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (rc != ECHO_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != ECHO_OK ? rc : cuda_fail(e, "end capture");
  }
  cudaGraphExec_t x = nullptr;
  e = cudaGraphInstantiate(&x, g, 0);
  if (e != cudaSuccess) {
    cudaGraphDestroy(g);
    return cuda_fail(e, "graph instantiation");
  }
  echo_step_graph *h = new (std::nothrow) echo_step_graph;
  if (!h) {
    cudaGraphExecDestroy(x);
    cudaGraphDestroy(g);
    set_error("out of host memory");
    return ECHO_EINVAL;
  }
  h->graph = g;
  h->exec = x;
  h->args = *a;
  *out = h;
  return ECHO_OK;
}

int echo_step_graph_launch(echo_step_graph *h, const void *q_host, const float *w_host, void *stream,
                           int32_t wait) {
  g_err[0] = 0;
  REQUIRE(h, "graph is NULL");
  REQUIRE((q_host == nullptr) == (w_host == nullptr), "give both q_host and w_host, or neither");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (q_host) TRY(copy_step_inputs(&h->args, q_host, w_host, s));
  const cudaError_t e = cudaGraphLaunch(h->exec, s);
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  return wait ? wait_stream(s) : ECHO_OK;
}

int echo_step_graph_destroy(echo_step_graph *h) {
  g_err[0] = 0;
  if (!h) return ECHO_OK;
  const cudaError_t e1 = cudaGraphExecDestroy(h->exec);
  const cudaError_t e2 = cudaGraphDestroy(h->graph);
  delete h;
  if (e1 != cudaSuccess) return cuda_fail(e1, "graph destroy");
  return e2 == cudaSuccess ? ECHO_OK : cuda_fail(e2, "graph destroy");
}

}  // extern "C"
