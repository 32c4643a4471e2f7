/*
 * echo.h -- C ABI of the GB300 (sm_103a) ECHO decode step.
 *
 * One layer of a DeepSeek-V3.2-style sparse-attention decode step, as the ECHO
 * review describes it (marsggbo.github.io, "OSDI'26 | ECHO: sparse attention saves
 * compute but blows up HBM", section 4 step list):
 *   indexer score (with the fused lossless prefetch) -> exact top-k ->
 *   guaranteed recall through the graph-friendly cache manager -> EMA of the k-th
 *   score, optionally preceded by the write-through append of the new token.
 *
 * Conventions for every call:
 *   - Returns ECHO_OK (0) or a negative-free error code below.  Argument errors are
 *     detected on the host before anything is enqueued (ECHO_EINVAL); a failing
 *     CUDA launch gives ECHO_ECUDA.  echo_last_error_string() describes the last
 *     error of the calling thread.
 *   - Work is enqueued on the caller's stream (`stream` is a cudaStream_t, NULL =
 *     the legacy default stream).  No call synchronises, allocates device or host
 *     memory, or reads device memory on the host, so every call can be captured
 *     into a CUDA graph (the first call of a process also sets kernel attributes;
 *     make one call outside capture first).  The exceptions are the host-input
 *     calls echo_decode_step_host and echo_step_graph_* (they may wait for their
 *     stream, and the graph calls own a captured graph).
 *   - The caller owns all memory.  Device pointers come from cudaMalloc or
 *     PyTorch; the host KV pool must be pinned and mapped (cudaHostAlloc with
 *     cudaHostAllocMapped, or any pinned allocation under unified addressing) and is
 *     passed as its device-accessible pointer; kernels read and write it directly.
 *   - Outcomes found on the device are OR-ed into the caller's `dev_status` int32
 *     (device memory) as ECHO_DEV_* bits; the caller clears it and reads it after
 *     synchronising.
 *   - "INF" in the residency maps is ECHO_INF (INT32_MAX).
 */
#ifndef ECHO_GB300_H
#define ECHO_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes -------------------------------------------------------- */
#define ECHO_OK 0
#define ECHO_EINVAL 1     /* bad argument (size, alignment, pointer kind)     */
#define ECHO_ECUDA 2      /* a CUDA runtime/driver call failed                */
#define ECHO_ENOTSUP 3    /* shape outside what the kernels support           */

/* ---- device status bits (OR-ed into *dev_status) ------------------------- */
#define ECHO_DEV_POOL_EXHAUSTED 1   /* too few evictable slots: rows left out   */
#define ECHO_DEV_BAD_INDEX 2        /* an index outside its array was skipped   */
#define ECHO_DEV_WAIT_TIMEOUT 4     /* a pipeline wait gave up (kernel aborted) */
#define ECHO_DEV_PREFETCH_CAP_HIT 8 /* info: prefetch candidates exceeded the cap
                                       (staging) or the reserve (direct to slot) */
#define ECHO_DEV_INVARIANT 16       /* echo_pool_validate found a broken invariant */

#define ECHO_INF 0x7fffffff
#define ECHO_H_INDEX 64      /* indexer heads            */
#define ECHO_D_INDEX 128     /* indexer head dim (e4m3)  */
#define ECHO_KV_ELEMS 576    /* latent KV per token: 512 + 64 rope, bf16 */
#define ECHO_KV_BYTES 1152

/*
 * One layer's GPU pool and its view of the host pool (section 5.1 metadata table;
 * GPU pool per layer, host pool per model).  All metadata arrays are device
 * memory; together they take 4*n_h + 13*n_g bytes (section 5.1 storage law).
 *   gpu_token_free      [n_g] uint8  GPUTokenFree: 1 = slot free
 *   gpu_token_priority  [n_g] int32  GPUTokenPriority: eviction clock, -1 when free
 *   gpu_indices_buffer  [n_g] int32  GPUIndicesBuffer: slots produced by the last
 *                                    allocate (or evict) call, -1 beyond
 *   gpu_token_to_host   [n_g] int32  GPUTokenToHost: INF when empty
 *   host_token_to_gpu   [n_h] int32  HostTokenToGPU: INF when not resident
 *   gpu_kv              [n_g][R] bf16  device KV pool, one row per slot
 *   host_kv             [n_h][R] bf16  pinned, mapped host pool (device pointer)
 *   counters            [4] int32 device: [0] free slots, [1] entries in use in
 *                       gpu_indices_buffer, [2..3] reserved
 *   row_elems           R, the bf16 elements of one row (the unit the metadata
 *                       tracks): 0 means 576, MLA's latent row of one token (512 +
 *                       64 rope).  Any multiple of 8 up to 65536 serves the
 *                       block-level / GQA variant (section 8: the cache manager
 *                       carries over to block-level sparsity by coarser metadata and
 *                       a KV-head dimension): a row is then one block of tokens of
 *                       one KV head (tokens x head dim x {K, V}), and a selection
 *                       per (request, KV head) folds the KV heads into the request
 *                       dimension of the calls below.  The cache-manager calls
 *                       (init, allocate, evict, recall without a stage, append)
 *                       take any R; the calls that prefetch (indexer or prefill
 *                       with a pool, recall with a stage, the decode step) need
 *                       R = 576.
 * Slots and host rows are plain indices; the pool is consistent when
 * host_token_to_gpu[gpu_token_to_host[s]] == s for every occupied slot s.
 */
typedef struct echo_pool {
    int32_t n_g;
    int32_t n_h;
    uint8_t *gpu_token_free;
    int32_t *gpu_token_priority;
    int32_t *gpu_indices_buffer;
    int32_t *gpu_token_to_host;
    int32_t *host_token_to_gpu;
    uint16_t *gpu_kv;
    uint16_t *host_kv;
    int32_t *counters;
    int32_t row_elems;
} echo_pool;

/*
 * Device scratch of the cache-manager calls, sized by echo_workspace_bytes() for
 * a pool of n_g slots and at most max_rows selected rows per call
 * (B * n_q * k for recall; B for append; n for allocate).  Initialise once with
 * echo_workspace_init(); every call leaves it initialised again.  One workspace
 * serves calls that run one after another on one stream.
 */
typedef struct echo_workspace {
    void *base;       /* device memory, 256-byte aligned */
    size_t bytes;
    int32_t n_g;
    int32_t max_rows;
} echo_workspace;

/*
 * Cumulative counters (device memory, int64 each; the caller zeroes them).
 * selected/unique_rows/hits/misses count the selected rows of a recall (hits and
 * misses after de-duplication, residency when the recall starts: a row the
 * direct-to-slot prefetch placed is a hit); recalled = misses that got a slot;
 * unrecalled = misses left out (pool exhausted); evicted = slots freed; staged =
 * rows the prefetch copied; staged_used = recalled rows taken from the staging
 * area (staging) or prefetched rows that were selected (direct to slot); appended
 * = tokens written through by append.
 */
typedef struct echo_stats {
    int64_t steps, selected, unique_rows, hits, misses, recalled, unrecalled, evicted,
        staged, staged_used, appended;
} echo_stats;

/*
 * Where the fused prefetch puts rows (section 6.1 intra-query prefetch; the page
 * leaves the landing place open).  Two modes:
 *
 * Staging (reserve == NULL): a staging area in HBM; the recall copies the staged
 * rows that were selected into their slots, the rest are dropped.
 *   rows        [B][stride][576] bf16 device
 *   host_row    [B][stride] int32 device  host row held by each staged row
 *   count       [B] int32 device          prefetch counter of each request; must
 *                                         be 0 before the indexer runs; the recall
 *                                         resets it to 0
 *   stride      rows reserved per request
 *   cap_div     request b stages at most min(stride, ceil(ctx_len[b] / cap_div))
 *               rows (cap proportional to the context length)
 *
 * Direct to slot (reserve != NULL): prefetched rows go straight into GPU-pool slots
 * that the previous recall set aside, and stay resident whether selected or not.
 * Reserved slots have gpu_token_free = 0, gpu_token_priority = -2 and no host row;
 * allocate, evict and append leave them alone.  Each prefetched row takes the next
 * ticket of reserve_ctl[0]; ticket t < reserve_ctl[1] puts it into slot reserve[t]
 * (host_token_to_gpu is claimed with a compare-and-swap, so a row is placed once).
 * A recall with this stage then counts the filled slots (stats staged; the
 * selected ones in staged_used), gives the unselected ones priority = clock,
 * returns the unused reserve to the free slots, evicts for its misses plus
 * reserve_cap more slots (as far as evictable slots go), and sets aside the
 * reserve_cap lowest-index free slots left after its allocation as the next
 * reserve.  A recall with reserve_cap = 0 returns the whole reserve.  An indexer
 * call with a direct stage must be followed by a recall with the same stage.
 *   reserve     int32 device, as long as the largest reserve_cap used with it:
 *               the reserved slots, in ticket order
 *   reserve_ctl [2] int32 device   [0] tickets drawn, [1] reserve length; zero both
 *                                  before first use
 *   reserve_cap slots each recall sets aside (0 <= reserve_cap <= n_g); may change
 *               between recalls
 *   count       may be NULL; rows, host_row, stride and cap_div are not used
 *
 * Both modes:
 *   flags       0, or ECHO_PREFETCH_WHILE_SCORING: the decode indexer's prefetch reads
 *               no host row for a candidate still queued when its CTA has scored its
 *               last tile, and takes no candidate from the last two tiles each of its
 *               epilogue warpgroups scores when a group scores at least eight (those
 *               copies would only lengthen the kernel; the recall fetches the rows that
 *               are selected).  Which rows are
 *               prefetched then depends on timing; selections, slots of selected rows
 *               and their bytes do not.
 *               The prefill indexer ignores the flag.
 */
#define ECHO_PREFETCH_WHILE_SCORING 1

typedef struct echo_stage {
    uint16_t *rows;
    int32_t *host_row;
    int32_t *count;
    int32_t stride;
    int32_t cap_div;
    int32_t *reserve;
    int32_t *reserve_ctl;
    int32_t reserve_cap;
    int32_t flags;
} echo_stage;

/*
 * Lightning-indexer score (section 2 "DSA indexer"; section 6.3 fused kernel):
 *   scores[b][j][p] = sum_{h<64} w[b][j][h] * ReLU( sum_{d<128} q[b][j][h][d] * k_index[b][p][d] )
 * for p < ctx_len[b] - (n_q - 1 - j) (query j of a request scoring n_q new
 * tokens sees that many keys); other entries of `scores` are left untouched.
 *   q        [B][n_q][64][128] e4m3 device, 16-byte aligned
 *   w        [B][n_q][64] fp32 device
 *   k_index  [B][L_max][128] e4m3 device, 16-byte aligned (the indexer K cache)
 *   ctx_len  [B] int32 device, 0 <= ctx_len[b] <= L_max
 *   scores   [B][n_q][L_max] fp32 device
 * FP8 products accumulate in the tensor cores' fp32 accumulator; the ReLU and the
 * weighted head sum run in fp32.
 * Fused prefetch (enabled when s_hat != NULL; section 6.1): a token whose score
 * exceeds s_hat[b][j] for some j and whose host row req_to_host[b][p] is not
 * resident takes a ticket from stage->count[b]; tickets below the cap copy the
 * host row into stage->rows[b][ticket] and record it in stage->host_row.  With a
 * direct-to-slot stage the row goes into the next reserved slot instead (see
 * echo_stage) and the pool's maps are updated.  The prefetch never changes what
 * is selected.  Needs pool (read-only in staging mode), req_to_host [B][L_max]
 * int32 device, stage.
 */
typedef struct echo_indexer_args {
    const uint8_t *q;
    const float *w;
    const uint8_t *k_index;
    const int32_t *ctx_len;
    int32_t B, n_q, L_max;
    float *scores;
    /* fused prefetch, all optional */
    const float *s_hat;
    const int32_t *req_to_host;
    const echo_pool *pool;
    const echo_stage *stage;
    int32_t *dev_status;
} echo_indexer_args;

int echo_indexer_score(const echo_indexer_args *args, void *stream);

/*
 * Indexer score of a prefill chunk with the fused inter-query prefetch (section 6.2;
 * section 6.3, prefill kernel).  Request b scores its last C tokens as queries: query
 * i sees ctx_len[b] - (C - 1 - i) keys (the chunk's own k^I rows are already in
 * k_index), and scores[b][i][p] is the formula of echo_indexer_score; other entries
 * are left untouched.  Queries are taken in blocks of 4 (one 4 x 64-head tensor-core
 * operand); each CTA owns whole blocks and all their keys.
 * Approximate top-k (s_shift != NULL): every score of query i is shifted by the
 * predicted k-th score, x = s - s_shift[b] (fp32), and binned by the top 8 bits of
 * x's order-preserving 32-bit key (bin 255 = the largest values); the top j bins with
 * S_255 + ... + S_{256-j} <= k are taken, bin 255 - j is the threshold bin
 * (thr_bin[b][i], -1 when all bins fit) and subset_n[b][i] counts the taken scores.
 * When a block is finished, the tokens some query of the block puts above its
 * threshold bin whose host row is not resident are prefetched as in the decode
 * indexer (staging or direct to slot, see echo_stage; once per block, a staged row
 * may repeat across blocks), while the following blocks are being scored.  Without
 * a stage only thr_bin / subset_n are produced.
 *   q        [B][C][64][128] e4m3 device, 16-byte aligned
 *   w        [B][C][64] fp32 device, 16-byte aligned
 *   k_index  [B][L_max][128] e4m3 device, 16-byte aligned
 *   ctx_len  [B] int32 device, 0 <= ctx_len[b] <= L_max (a context shorter than C
 *            gives the first queries no keys)
 *   scores   [B][C][L_max] fp32 device
 *   s_shift  [B] fp32 device, optional; k >= 1 with it
 *   thr_bin, subset_n  [B][C] int32 device, optional
 *   req_to_host [B][L_max] int32 device, pool, stage: optional (prefetch)
 */
typedef struct echo_prefill_args {
    const uint8_t *q;
    const float *w;
    const uint8_t *k_index;
    const int32_t *ctx_len;
    int32_t B, C, L_max;
    float *scores;
    const float *s_shift;
    int32_t k;
    int32_t *thr_bin;
    int32_t *subset_n;
    const int32_t *req_to_host;
    const echo_pool *pool;
    const echo_stage *stage;
    int32_t *dev_status;
} echo_prefill_args;

int echo_prefill_indexer_score(const echo_prefill_args *args, void *stream);

/*
 * Exact top-k per (b, j) row of `scores` over its first
 * ctx_len[b] - (n_q - 1 - j) entries (section 2: top-k with k = 2048).  Ties at the
 * k-th value go to the lower token index.  sel[b][j][0..k) lists the selected
 * token indices in ascending order, -1 padded when fewer than k tokens exist;
 * kth[b][j] is the min(k, L)-th largest score (-inf for an empty row).
 *   scores [B][n_q][L_max] fp32 device (no NaN); sel [B][n_q][k] int32; kth [B][n_q] fp32
 * Limits: 1 <= k <= 8192, L_max <= 360448, 1 <= n_q <= 65536 (the queries of a
 * prefill chunk are rows too).
 */
int echo_select_topk(const float *scores, const int32_t *ctx_len, int32_t B, int32_t n_q,
                     int32_t L_max, int32_t k, int32_t *sel, float *kth, void *stream);

/* Sizes and initialisation of the cache-manager scratch. */
int echo_workspace_bytes(int32_t n_g, int32_t max_rows, size_t *bytes);
int echo_workspace_init(const echo_workspace *ws, void *stream);

/* Empty pool: free = 1, priority = -1, indices buffer = -1, both maps = INF,
   counters = {n_g, 0}.  Does not touch gpu_kv or host_kv. */
int echo_pool_init(const echo_pool *pool, void *stream);

/*
 * Allocate (section 5.2): give host_idx[0..n) GPU slots, n = *n_dev (device),
 * n <= max_n.  The i-th valid row takes the i-th lowest free slot (the atomic
 * tickets of the page taken in slot order); the slot's priority becomes `clock`
 * (or *clock_dev when clock_dev != NULL), both maps are set, out_slots[i] = slot
 * and gpu_indices_buffer[0..granted) lists the slots.  Rows already resident,
 * repeated or out of range get -1 and ECHO_DEV_BAD_INDEX; rows beyond the free
 * slots get -1 and ECHO_DEV_POOL_EXHAUSTED.  No KV bytes move.
 */
int echo_pool_alloc(const echo_pool *pool, const echo_workspace *ws, const int32_t *host_idx,
                    const int32_t *n_dev, int32_t max_n, int32_t clock, const int32_t *clock_dev,
                    int32_t *out_slots, int32_t *dev_status, void *stream);

/*
 * Free (section 5.2): evict n = *n_needed_dev slots with the smallest
 * (priority, slot) among occupied slots whose priority is below the clock
 * (selected tokens carry priority == clock, which protects them).  Sets free = 1,
 * priority = -1, HostTokenToGPU = INF, GPUTokenToHost = INF; gpu_indices_buffer
 * lists the evicted slots in ascending order.  No KV bytes move.  Fewer evictable
 * slots than asked: all of them go and ECHO_DEV_POOL_EXHAUSTED is set.
 */
int echo_pool_evict(const echo_pool *pool, const echo_workspace *ws, const int32_t *n_needed_dev,
                    int32_t clock, const int32_t *clock_dev, int32_t *dev_status, void *stream);

/*
 * Guaranteed recall (section 4 step list; section 5.2 "Recall"):
 *   (i) map sel[b][j][i] to host rows req_to_host[b][p], first occurrence in
 *   (b, j, i) order; (ii) resident rows: priority = clock; (iii) evict
 *   max(0, misses - free) slots; (iv) allocate the misses in order; (v) copy each
 *   recalled row from the staging area when the prefetch staged it this step,
 *   else from host_kv, into gpu_kv; (vi) out_slot[b][j][i] = slot of sel[b][j][i],
 *   -1 for padding and for rows left out when the pool is exhausted.
 *   sel [B][n_q][k] int32 device; req_to_host [B][L_max] int32 device;
 *   stage optional (NULL: nothing staged); stats optional (device echo_stats).
 * B * n_q * k must not exceed ws->max_rows.
 */
int echo_prefetch_recall(const echo_pool *pool, const echo_workspace *ws, const int32_t *sel,
                         const int32_t *req_to_host, const int32_t *ctx_len, int32_t B, int32_t n_q,
                         int32_t k, int32_t L_max, const echo_stage *stage, int32_t clock,
                         const int32_t *clock_dev, int32_t *out_slot, echo_stats *stats,
                         int32_t *dev_status, void *stream);

/*
 * The guaranteed recall above, for callers that cannot allocate device memory:
 * it uses no caller workspace and makes no allocation of any kind (no cudaMalloc,
 * no cudaFree, no allocating library call).  The page has no counterpart of this
 * call; it exists for callers such as a memory-planned serving runtime that has
 * already divided all device memory between weights and KV pools and may not grow
 * it at run time, or a plugin behind a foreign-language boundary that is handed
 * buffers but no allocator.
 * Its scratch is one fixed array inside the library per device (4 MiB, held by
 * every GPU that loads the library until the process exits), laid out for pools of
 * at most 262144 slots and at most 32768 selected entries (B * n_q * k); larger
 * calls return ECHO_EINVAL with a message.  A call made outside stream capture looks
 * up the array's device address on the current device (so a context re-created after
 * cudaDeviceReset is served too); a call made while the stream is capturing reuses the
 * address found by the last such lookup on that device, so make the first call on each
 * device before any stream capture.  Devices 0..63 are served (ECHO_ENOTSUP beyond).  Every
 * call re-initialises the array before using it (one extra small kernel), and all
 * calls share it: calls whose work overlaps on the GPU (other streams, other
 * threads) race and must not be issued.  Arguments and results as in
 * echo_prefetch_recall.
 */
int echo_prefetch_recall_noalloc(const echo_pool *pool, const int32_t *sel, const int32_t *req_to_host,
                                 const int32_t *ctx_len, int32_t B, int32_t n_q, int32_t k, int32_t L_max,
                                 const echo_stage *stage, int32_t clock, const int32_t *clock_dev,
                                 int32_t *out_slot, echo_stats *stats, int32_t *dev_status, void *stream);

/*
 * Write-through append of the token each request generated (section 2 "offload";
 * section 5.2 "Free" notes the host copy is made at generation): for request b,
 * p = ctx_len[b]; new_kv[b] is written to host row req_to_host[b][p] and to a newly
 * allocated GPU slot (priority = clock, evicting first if the pool is short),
 * new_k_index[b] to k_index[b][p]; then ctx_len[b] = p + 1.
 *   new_kv [B][R] bf16 device (R = the pool's row_elems); new_k_index [B][128] e4m3 device.
 */
int echo_append(const echo_pool *pool, const echo_workspace *ws, uint8_t *k_index, int32_t *ctx_len,
                const int32_t *req_to_host, int32_t B, int32_t L_max, const uint16_t *new_kv,
                const uint8_t *new_k_index, int32_t clock, const int32_t *clock_dev,
                echo_stats *stats, int32_t *dev_status, void *stream);

/*
 * EMA of the k-th score (section 6.1): s_hat = alpha*s_hat + (1-alpha)*kth in fp32
 * (multiply, multiply, add, each rounded); s_hat = +inf (the start value, no
 * prefetch) takes kth directly; a non-finite kth (empty row) leaves s_hat as is.
 */
int echo_ema_update(float *s_hat, const float *kth, int32_t n, float alpha, void *stream);

/* The same EMA reading kth[i * kth_stride] (a prefill chunk updates its request's
   prediction from the k-th score of the chunk's last query: kth + C - 1, stride C). */
int echo_ema_update_strided(float *s_hat, const float *kth, int32_t n, int32_t kth_stride, float alpha,
                            void *stream);

/*
 * Sparse MLA decode over the selected rows (section 2: MLA's latent row of d_c = 512 +
 * 64 rope dims is shared by all 128 heads; the indexer's top-k feeds sparse attention).
 * With the up-projections absorbed, head h of query token (b, j) attends over the
 * rows out_slot[b][j][0..k) names in the GPU pool:
 *   s_i = scale * q[b][j][h] . gpu_kv[slot_i]            (576 dims, fp32 accumulate)
 *   out[b][j][h] = sum_i softmax(s)_i * gpu_kv[slot_i][0..512)
 *   lse[b][j][h] = log sum_i exp(s_i)
 * Entries with slot < 0 are skipped (slot >= n_g: also ECHO_DEV_BAD_INDEX); a head
 * with no row gives out = 0, lse = -inf.  The softmax weights enter the value product
 * rounded to bf16 (the tensor cores' operand type); everything else is fp32.
 *   q       [B][n_q][128][576] bf16 device, 16-byte aligned
 *   gpu_kv  [n_g][576] bf16 device (the pool's rows)
 *   out_slot [B][n_q][k] int32 device, 1 <= k <= 8192
 *   out     [B][n_q][128][512] fp32 device;  lse [B][n_q][128] fp32 device
 *   workspace  device, 256-byte aligned, echo_mla_workspace_bytes() bytes
 * Launches 2 kernels (one CTA per 128 selected rows of each query token, then the
 * merge of their partial results).
 */
typedef struct echo_mla_args {
    const uint16_t *q;
    const uint16_t *gpu_kv;
    int32_t n_g;
    const int32_t *out_slot;
    int32_t B, n_q, k;
    float scale;
    float *out;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    int32_t *dev_status;
} echo_mla_args;

int echo_mla_workspace_bytes(int32_t B, int32_t n_q, int32_t k, size_t *bytes);
int echo_sparse_mla_decode(const echo_mla_args *args, void *stream);

/* Stages of echo_decode_step, in order (timing events are recorded before each
   stage and after the last).  The EMA is computed by the recall's last kernel, so
   the ECHO_STAGE_EMA interval is empty; the constant is kept for the event layout. */
#define ECHO_STAGE_APPEND 0
#define ECHO_STAGE_INDEXER 1
#define ECHO_STAGE_TOPK 2
#define ECHO_STAGE_RECALL 3
#define ECHO_STAGE_EMA 4
#define ECHO_NUM_STAGES 5

/*
 * One layer's decode step, every stage on the device (section 4 step list):
 *   [append] -> indexer score + fused prefetch -> top-k -> guaranteed recall -> EMA.
 * Fields as in the single calls.  new_kv == NULL skips the append.  s_hat may be
 * NULL (no prefetch, no EMA); prefetch also needs stage.  When clock_dev != NULL
 * the kernels read the clock there and, if advance_clock != 0, the recall advances
 * it by one, so one captured graph can be replayed step after step.  All arguments
 * are checked before the first launch: a rejected step enqueues nothing.
 * Launches: 3 kernels (indexer; top-k, which also makes the recall's claims; the
 * cooperative cache-manager kernel, which also updates the EMA), the last two as
 * programmatic dependent launches; plus 2 for the append (write-through kernel,
 * cache-manager kernel).  stage_events: optional array of
 * ECHO_NUM_STAGES + 1 cudaEvent_t (timing-enabled) recorded around the stages
 * (as external event nodes under stream capture, plain records otherwise).
 */
typedef struct echo_step_args {
    const echo_pool *pool;
    const echo_workspace *ws;
    const echo_stage *stage;
    const uint8_t *q;
    const float *w;
    uint8_t *k_index;
    int32_t *ctx_len;
    const int32_t *req_to_host;
    int32_t B, n_q, L_max, k;
    float *scores;
    int32_t *sel;
    float *kth;
    int32_t *out_slot;
    float *s_hat;
    float alpha;
    const uint16_t *new_kv;
    const uint8_t *new_k_index;
    int32_t clock;
    int32_t *clock_dev;
    int32_t advance_clock;
    echo_stats *stats;
    int32_t *dev_status;
    void **stage_events;
} echo_step_args;

int echo_decode_step(const echo_step_args *args, void *stream);

/*
 * The same step with its per-step inputs taken from host memory, for callers whose
 * query and head weights are produced on the host.  q_host holds B * n_q * 64 * 128
 * e4m3 bytes laid out as args->q, w_host B * n_q * 64 floats laid out as args->w;
 * both are copied on `stream` into args->q and args->w (one copy when w follows q
 * directly in both buffers), then the step runs exactly as echo_decode_step.  The host
 * buffers should be pinned (pageable memory makes the copy synchronous) and must stay
 * unchanged until the copy has run.  wait != 0: the call returns once the stream has
 * finished the step, so results the kernels wrote into pinned host memory (out_slot,
 * dev_status) can be read at once.  Unlike the calls above, this one may synchronise
 * (wait != 0).  Errors: as echo_decode_step, plus ECHO_EINVAL for a NULL q_host or
 * w_host and ECHO_ECUDA when the copy or the synchronisation fails.
 */
int echo_decode_step_host(const echo_step_args *args, const void *q_host, const float *w_host, void *stream,
                          int32_t wait);

/*
 * A decode step captured once into a CUDA graph owned by the library, then launched
 * step after step: the serving loop's form of echo_decode_step_host.  create checks
 * args as echo_decode_step does, requires the device clock (clock_dev != NULL; with
 * advance_clock != 0 each launch is the next step) and no stage events, and captures
 * the step's launches on a stream of its own (nothing runs).  The graph keeps the
 * pointers in args: every buffer must outlive it.  launch copies q_host / w_host (as
 * in echo_decode_step_host; both NULL: the inputs are already in args->q and args->w)
 * and launches the graph on `stream`, waiting for it when wait != 0.  destroy frees
 * the graph (NULL is accepted).  create allocates host memory and graph objects; a
 * failed create returns no graph (*out = NULL).
 */
typedef struct echo_step_graph echo_step_graph;
int echo_step_graph_create(const echo_step_args *args, echo_step_graph **out);
int echo_step_graph_launch(echo_step_graph *graph, const void *q_host, const float *w_host, void *stream,
                           int32_t wait);
int echo_step_graph_destroy(echo_step_graph *graph);

/*
 * Metadata invariants of one pool (section 5.1 metadata table; section 5.2 "Free":
 * a freed slot has free = 1, priority = -1 and no host row).  Every slot is in one
 * state:
 *   free       gpu_token_free = 1, priority = -1, gpu_token_to_host = INF
 *   occupied   free = 0, priority >= 0 (or the prefetch's mark -3 between a
 *              direct-to-slot indexer and its recall), gpu_token_to_host = h in
 *              [0, n_h) with host_token_to_gpu[h] = s
 *   reserved   free = 0, priority = -2, gpu_token_to_host = INF (direct to slot)
 * and every host row is absent (host_token_to_gpu = INF) or maps to a slot that maps
 * back.  counters[0] must equal the number of free slots; with a direct-to-slot
 * stage the reserve's first reserve_ctl[1] entries must be reserved slots and no
 * other slot may be.  Meant for quiescent points (between steps): inside a recall
 * the maps hold claim marks by design.
 * report receives ECHO_VAL_COUNT int32 values (indices below): the first five count
 * violations, the next four the slots / rows seen in each state, the last one is the
 * reserve's index balance (a non-zero balance counts as a reserve violation).
 */
#define ECHO_VAL_SLOT_STATE 0 /* slots whose free flag, priority and host row disagree  */
#define ECHO_VAL_SLOT_MAP 1   /* occupied slots whose host row maps elsewhere           */
#define ECHO_VAL_ROW_MAP 2    /* resident rows whose slot is out of range or elsewhere  */
#define ECHO_VAL_COUNTER 3    /* 1 when counters[0] differs from the free slots         */
#define ECHO_VAL_RESERVE 4    /* reserve entries that are not reserved slots, plus 1
                                 when the reserved slots and the reserve's length differ */
#define ECHO_VAL_FREE 5       /* free slots                                            */
#define ECHO_VAL_OCCUPIED 6   /* occupied slots                                        */
#define ECHO_VAL_RESERVED 7   /* reserved slots                                        */
#define ECHO_VAL_RESIDENT 8   /* host rows with a slot                                 */
#define ECHO_VAL_BALANCE 9    /* sum of the reserved slots' indices minus the sum of
                                 the reserve's entries (mod 2^32): 0 unless the reserve
                                 repeats a slot and leaves another out               */
#define ECHO_VAL_COUNT 10

/*
 * The check on the device, in stream order: report [ECHO_VAL_COUNT] int32 device
 * memory (overwritten); ECHO_DEV_INVARIANT is OR-ed into *dev_status when a violation
 * count is non-zero.  stage: NULL, or a direct-to-slot stage whose reserve is checked.
 * The reserve array is read only up to stage->reserve_cap entries (its length by the
 * echo_stage contract); a recorded length above that counts as a reserve violation.
 * Launches 2 kernels after clearing report; capturable.
 */
int echo_pool_validate(const echo_pool *pool, const echo_stage *stage, int32_t *report, int32_t *dev_status,
                       void *stream);

/*
 * The same check over HOST copies of the arrays (every pointer in *pool_host is a
 * host pointer; gpu_kv and host_kv are not read), for a snapshot taken with
 * cudaMemcpy or for tools without a GPU.  reserve: NULL or reserve_len host int32.
 * Fills report [ECHO_VAL_COUNT] (host) and returns ECHO_DEV_INVARIANT when a
 * violation was found, else 0 (a negative value: bad arguments).
 */
int echo_pool_validate_host(const echo_pool *pool_host, const int32_t *reserve, int32_t reserve_len,
                            int32_t *report);

/*
 * Self-test of the failure detection (no counterpart on the pages): launches a
 * kernel whose wait nothing will satisfy -- which = 0: an mbarrier wait (the wait the
 * indexer's roles use), which = 1: a grid barrier of a cooperative launch that one CTA
 * never reaches (the barrier the cache-manager kernel uses).  The wait gives up after
 * one second, ECHO_DEV_WAIT_TIMEOUT is OR-ed into *dev_status (device memory) and
 * every CTA returns; the context stays usable.  Takes about one second of GPU time.
 */
int echo_selftest_wait_timeout(int32_t which, int32_t *dev_status, void *stream);

/* Description of the calling thread's last error ("" if none). */
const char *echo_last_error_string(void);

/* Library version, (major << 16) | minor (1.1: echo_stage's direct-to-slot fields;
   1.2: echo_prefill_indexer_score, echo_ema_update_strided, n_q up to 65536 in
   top-k and recall; 1.3: echo_sparse_mla_decode; 1.4: echo_pool.row_elems,
   echo_stage.flags; 1.5: echo_pool_validate, echo_pool_validate_host). */
int32_t echo_version(void);

/* Storage law of the metadata arrays of one pool (section 5.1): 4*n_h + 13*n_g. */
int64_t echo_metadata_bytes(int64_t n_h, int64_t n_g);

#ifdef __cplusplus
}
#endif
#endif /* ECHO_GB300_H */
