/*
 * echo_oracle.c -- plain, slow, single-threaded CPU oracle of the ECHO decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load or call this code.  It shares no code
 * with the CUDA library: no header, helper or table of the CUDA path is used here.
 *
 * Source of every rule: the ECHO review page (marsggbo.github.io,
 * "OSDI'26 | ECHO: sparse attention saves compute but blows up HBM").
 *   - section 2 "DSA indexer": index score s(t,s) = sum_h w_{h,t} ReLU(q_{h,t} . k_s),
 *     H_index = 64, d_index = 128, FP8 q/k; top-k with k = 2048.
 *   - section 5.1, metadata table: GPUTokenFree, GPUTokenPriority (-1 when free),
 *     GPUIndicesBuffer, GPUTokenToHost (inf = empty), HostTokenToGPU (inf = absent);
 *     storage law 4*N_H + 13*N_G bytes.
 *   - section 5.2, "Allocate": free-slot threads draw atomicAdd tickets; tickets below
 *     `size` win; priority raised from -1; both maps set; indices go to
 *     GPUIndicesBuffer with -1 for invalid entries.
 *   - section 5.2, "Free": protect the step's selected tokens, arg-top-k of the lowest
 *     priorities, scatter free / ToHost = inf / HostToGPU = inf; no data moves.
 *   - section 5.2, "Recall": look up HostTokenToGPU of the selected host rows (inf =
 *     missing), free + allocate, set both maps, copy the KV from host to GPU.
 *   - section 6.1: EMA of the k-th score, s_hat(t+1) = alpha s_hat(t) + (1-alpha) s(t),
 *     alpha = 0.5; tokens whose score exceeds the prediction are prefetched; a global
 *     counter caps the prefetch count in proportion to the context length; the final
 *     selection never depends on the prediction (lossless).
 *
 * Readings where the page is silent (each is listed in the design notes):
 *   R1 ReLU is applied to the dot product q.k (the page prints a comma).
 *   R2 q/k are raw e4m3 codes with no scale factors.
 *   R3 top-k ties at the k-th value go to the lower token index; output is in
 *      ascending token index, padded with -1; kth = the min(k, L)-th largest score,
 *      -inf when L == 0.
 *   R5 the prefetch test is strict (score > s_hat); s_hat starts at +inf (no
 *      prefetch) and takes the first observed kth directly.
 *   R6 prefetch cap per request = min(stage rows, ceil(L / cap_div)).
 *   R8 allocation tickets follow ascending slot order unless an explicit ticket
 *      permutation is given (that reproduces the page's worked example).
 *   R9 priority is a step clock: selected -> clock; eviction takes the smallest
 *      (priority, slot) among occupied slots with priority < clock.
 *   R10 exactly max(0, misses - free) slots are evicted; if too few are evictable the
 *      status gets POOL_EXHAUSTED and the misses beyond capacity stay unrecalled.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_INF INT32_MAX
/* priority of a slot set aside for the direct-to-slot prefetch: not free, not
   evictable, not mapped */
#define ORC_RESERVED (-2)

enum {
    ORC_POOL_EXHAUSTED = 1,
    ORC_BAD_INDEX = 2,
    ORC_PREFETCH_CAP_HIT = 8,
};

/* ------------------------------------------------------------------------- */
/* FP8 e4m3 (the "fn" variant: no infinities, 0x7F/0xFF are NaN)              */
/* ------------------------------------------------------------------------- */

/* value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0, (-1)^s * 2^-6 * (m/8) for e == 0 */
double orc_e4m3_value(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* Lightning-indexer score (section 2, "DSA indexer")                         */
/* ------------------------------------------------------------------------- */

/* number of keys query j of a request with context L may see: causal over
   L - (n_q - 1 - j) tokens (multi-token prediction scores n_q new tokens) */
static int valid_len(int L, int n_q, int j)
{
    int v = L - (n_q - 1 - j);
    return v < 0 ? 0 : v;
}

/* score of token p for query (b, j), given the query already decoded to qd[H][D] */
static float score_token(const double *qd, const float *wb, const uint8_t *kp, int H, int D, double *kd)
{
    for (int d = 0; d < D; ++d)
        kd[d] = orc_e4m3_value(kp[d]);
    double s = 0.0;
    for (int h = 0; h < H; ++h) {
        /* e4m3 values are multiples of 2^-9 with |x| <= 448; with |x| <= 8 the
           products are multiples of 2^-18 below 2^6 and the 128-term sum stays far
           inside 53 bits, so this fp64 dot product is exact */
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qd[(size_t)h * D + d] * kd[d];
        double relu = dot > 0.0 ? dot : 0.0;
        s += (double)wb[h] * relu;
    }
    return (float)s;
}

static void decode_query(const uint8_t *q, int H, int D, double *qd)
{
    for (int i = 0; i < H * D; ++i)
        qd[i] = orc_e4m3_value(q[i]);
}

float orc_indexer_score_one(const uint8_t *q, const float *w, const uint8_t *k_index,
                            int n_q, int L_max, int H, int D, int b, int j, int p)
{
    double *qd = (double *)malloc(sizeof(double) * (size_t)H * D);
    double *kd = (double *)malloc(sizeof(double) * (size_t)D);
    decode_query(q + ((size_t)b * n_q + j) * H * D, H, D, qd);
    float s = score_token(qd, w + ((size_t)b * n_q + j) * H, k_index + ((size_t)b * L_max + p) * D, H, D, kd);
    free(qd);
    free(kd);
    return s;
}

/* scores[b][j][p] for p < valid_len(ctx_len[b], n_q, j); other entries untouched */
void orc_indexer_score(const uint8_t *q, const float *w, const uint8_t *k_index,
                       const int32_t *ctx_len, int B, int n_q, int L_max, int H, int D,
                       float *scores)
{
    double *qd = (double *)malloc(sizeof(double) * (size_t)H * D);
    double *kd = (double *)malloc(sizeof(double) * (size_t)D);
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < n_q; ++j) {
            int v = valid_len(ctx_len[b], n_q, j);
            decode_query(q + ((size_t)b * n_q + j) * H * D, H, D, qd);
            const float *wb = w + ((size_t)b * n_q + j) * H;
            for (int p = 0; p < v; ++p)
                scores[((size_t)b * n_q + j) * L_max + p] =
                    score_token(qd, wb, k_index + ((size_t)b * L_max + p) * D, H, D, kd);
        }
    free(qd);
    free(kd);
}

/* ------------------------------------------------------------------------- */
/* Exact top-k (section 2: top-k of the index scores, k = 2048)               */
/* ------------------------------------------------------------------------- */

typedef struct {
    float s;
    int32_t p;
} orc_sp;

static int cmp_score_desc_index_asc(const void *a, const void *b)
{
    const orc_sp *x = (const orc_sp *)a, *y = (const orc_sp *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->p > y->p) - (x->p < y->p);
}

static int cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* sel[b][j][0..k): selected token indices ascending, -1 padded; kth[b][j] */
void orc_select_topk(const float *scores, const int32_t *ctx_len, int B, int n_q, int L_max,
                     int k, int32_t *sel, float *kth)
{
    orc_sp *buf = (orc_sp *)malloc(sizeof(orc_sp) * (size_t)(L_max > 0 ? L_max : 1));
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < n_q; ++j) {
            size_t row = (size_t)b * n_q + j;
            int v = valid_len(ctx_len[b], n_q, j);
            for (int p = 0; p < v; ++p) {
                buf[p].s = scores[row * L_max + p];
                buf[p].p = p;
            }
            qsort(buf, (size_t)v, sizeof(orc_sp), cmp_score_desc_index_asc);
            int m = v < k ? v : k;
            int32_t *out = sel + row * k;
            for (int i = 0; i < m; ++i)
                out[i] = buf[i].p;
            qsort(out, (size_t)m, sizeof(int32_t), cmp_i32);
            for (int i = m; i < k; ++i)
                out[i] = -1;
            kth[row] = m > 0 ? buf[m - 1].s : -INFINITY;
        }
    free(buf);
}

/* ------------------------------------------------------------------------- */
/* Graph-friendly cache manager (section 5)                                   */
/* ------------------------------------------------------------------------- */

typedef struct {
    int32_t n_g, n_h, row_elems;
    uint8_t *GPUTokenFree;       /* [n_g] 1 = free                         */
    int32_t *GPUTokenPriority;   /* [n_g] -1 when free                     */
    int32_t *GPUIndicesBuffer;   /* [n_g] output of allocate/free, -1 pad  */
    int32_t *GPUTokenToHost;     /* [n_g] inf when empty                   */
    int32_t *HostTokenToGPU;     /* [n_h] inf when not resident            */
    uint16_t *gpu_kv;            /* [n_g][row_elems] bf16 bits             */
    uint16_t *host_kv;           /* [n_h][row_elems] bf16 bits             */
    int32_t n_free;              /* number of free slots                   */
    int32_t idx_count;           /* entries of GPUIndicesBuffer in use     */
} orc_pool;

typedef struct {
    int64_t steps, selected, unique_rows, hits, misses, recalled, unrecalled,
        evicted, staged, staged_used, appended;
} orc_stats;

void orc_pool_init(orc_pool *P)
{
    for (int s = 0; s < P->n_g; ++s) {
        P->GPUTokenFree[s] = 1;
        P->GPUTokenPriority[s] = -1;
        P->GPUIndicesBuffer[s] = -1;
        P->GPUTokenToHost[s] = ORC_INF;
    }
    for (int h = 0; h < P->n_h; ++h)
        P->HostTokenToGPU[h] = ORC_INF;
    P->n_free = P->n_g;
    P->idx_count = 0;
}

/* write list[0..n) into GPUIndicesBuffer, -1 over the rest of the old list */
static void set_indices_buffer(orc_pool *P, const int32_t *list, int n)
{
    for (int i = 0; i < n; ++i)
        P->GPUIndicesBuffer[i] = list[i];
    for (int i = n; i < P->idx_count; ++i)
        P->GPUIndicesBuffer[i] = -1;
    P->idx_count = n;
}

/*
 * Allocate (section 5.2): every slot thread reads GPUTokenFree; threads holding a
 * free slot take a ticket from a shared counter; tickets < size allocate.  The
 * ticket order is the order in which the atomicAdds land.  With tickets == NULL the
 * legal order where tickets follow ascending slot index is used; otherwise
 * tickets[s] is the ticket slot s drew (only free slots are read).
 * host_idx[i] goes to the slot holding ticket i.
 * Host rows already resident, duplicated or out of range get out_slots[i] = -1 and
 * BAD_INDEX.  If fewer slots are free than rows asked for, the rows beyond the free
 * count get -1 and POOL_EXHAUSTED.
 */
int orc_pool_alloc(orc_pool *P, const int32_t *host_idx, int n, int32_t clock,
                   const int32_t *tickets, int32_t *out_slots)
{
    int status = 0;
    /* rows that can take a slot, in order (first occurrence of each valid row) */
    int32_t *want = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t *want_pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    uint8_t *seen = (uint8_t *)calloc((size_t)P->n_h, 1);
    int size = 0;
    for (int i = 0; i < n; ++i) {
        int32_t h = host_idx[i];
        out_slots[i] = -1;
        if (h < 0 || h >= P->n_h || P->HostTokenToGPU[h] != ORC_INF || seen[h]) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        seen[h] = 1;
        want[size] = h;
        want_pos[size] = i;
        ++size;
    }
    free(seen);

    int32_t *won = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P->n_g > 0 ? P->n_g : 1));
    for (int i = 0; i < P->n_g; ++i)
        won[i] = -1;
    int counter = 0; /* the global atomicAdd counter */
    for (int s = 0; s < P->n_g; ++s) {
        if (!P->GPUTokenFree[s])
            continue;
        int ticket = tickets ? tickets[s] : counter;
        counter++;
        if (ticket < size)
            won[ticket] = s;
    }
    int granted = size < P->n_free ? size : P->n_free;
    if (granted < size)
        status |= ORC_POOL_EXHAUSTED;
    for (int t = 0; t < granted; ++t) {
        int s = won[t];
        int32_t h = want[t];
        P->GPUTokenFree[s] = 0;
        P->GPUTokenPriority[s] = clock;
        P->GPUTokenToHost[s] = h;
        P->HostTokenToGPU[h] = s;
        out_slots[want_pos[t]] = s;
    }
    P->n_free -= granted;
    set_indices_buffer(P, won, granted);
    free(won);
    free(want);
    free(want_pos);
    return status;
}

typedef struct {
    int32_t prio, slot;
} orc_ps;

static int cmp_prio_slot(const void *a, const void *b)
{
    const orc_ps *x = (const orc_ps *)a, *y = (const orc_ps *)b;
    if (x->prio != y->prio) return (x->prio > y->prio) - (x->prio < y->prio);
    return (x->slot > y->slot) - (x->slot < y->slot);
}

/*
 * Free (section 5.2).  Protection is the caller's step: selected tokens already
 * carry priority == clock, so only occupied slots with priority < clock compete.
 * Arg-top-k of the lowest (priority, slot), then scatter: free = 1, priority = -1,
 * HostTokenToGPU[GPUTokenToHost[s]] = inf, GPUTokenToHost[s] = inf.  The evicted
 * slots go to GPUIndicesBuffer in ascending slot order.  No KV bytes move.
 */
int orc_pool_evict(orc_pool *P, int n_needed, int32_t clock, int32_t *n_evicted)
{
    int status = 0;
    orc_ps *c = (orc_ps *)malloc(sizeof(orc_ps) * (size_t)(P->n_g > 0 ? P->n_g : 1));
    int nc = 0;
    for (int s = 0; s < P->n_g; ++s)
        if (!P->GPUTokenFree[s] && P->GPUTokenPriority[s] >= 0 && P->GPUTokenPriority[s] < clock) {
            c[nc].prio = P->GPUTokenPriority[s];
            c[nc].slot = s;
            ++nc;
        }
    int e = n_needed < 0 ? 0 : n_needed;
    if (e > nc) {
        status |= ORC_POOL_EXHAUSTED;
        e = nc;
    }
    qsort(c, (size_t)nc, sizeof(orc_ps), cmp_prio_slot);
    int32_t *victims = (int32_t *)malloc(sizeof(int32_t) * (size_t)(e > 0 ? e : 1));
    for (int i = 0; i < e; ++i)
        victims[i] = c[i].slot;
    qsort(victims, (size_t)e, sizeof(int32_t), cmp_i32);
    for (int i = 0; i < e; ++i) {
        int s = victims[i];
        int32_t h = P->GPUTokenToHost[s];
        P->GPUTokenFree[s] = 1;
        P->GPUTokenPriority[s] = -1;
        if (h >= 0 && h < P->n_h)
            P->HostTokenToGPU[h] = ORC_INF;
        P->GPUTokenToHost[s] = ORC_INF;
    }
    P->n_free += e;
    set_indices_buffer(P, victims, e);
    if (n_evicted)
        *n_evicted = e;
    free(victims);
    free(c);
    return status;
}

/*
 * Direct-to-slot prefetch (the pages' likely landing place for prefetched rows,
 * section 6.1 with the pool of section 5): a recall sets aside the reserve_cap
 * lowest-index slots that are free after it (evicting for them like for misses,
 * misses first); the next step's prefetch puts rows straight into them.  Reserved
 * slots are neither free nor evictable (allocate, evict and append leave them
 * alone); the next recall in direct mode returns the ones the prefetch left unused
 * to the free slots before it starts.
 */
/* occupied slots that may be evicted at this clock */
static int orc_evictable(const orc_pool *P, int32_t clock)
{
    int n = 0;
    for (int s = 0; s < P->n_g; ++s)
        n += !P->GPUTokenFree[s] && P->GPUTokenPriority[s] >= 0 && P->GPUTokenPriority[s] < clock;
    return n;
}

static int orc_reserve_release(orc_pool *P)
{
    int n = 0;
    for (int s = 0; s < P->n_g; ++s)
        if (!P->GPUTokenFree[s] && P->GPUTokenPriority[s] == ORC_RESERVED) {
            P->GPUTokenFree[s] = 1;
            P->GPUTokenPriority[s] = -1;
            P->GPUTokenToHost[s] = ORC_INF;
            ++n;
        }
    P->n_free += n;
    return n;
}

static int orc_reserve_take(orc_pool *P, int cap, int32_t *list)
{
    int n = 0;
    for (int s = 0; s < P->n_g && n < cap; ++s)
        if (P->GPUTokenFree[s]) {
            P->GPUTokenFree[s] = 0;
            P->GPUTokenPriority[s] = ORC_RESERVED;
            list[n++] = s;
        }
    P->n_free -= n;
    return n;
}

/* copy one latent-KV row host -> GPU pool */
static void copy_row(orc_pool *P, int32_t slot, const uint16_t *src)
{
    memcpy(P->gpu_kv + (size_t)slot * P->row_elems, src, sizeof(uint16_t) * (size_t)P->row_elems);
}

/*
 * The direct-to-slot prefetch of one step, as the GPU's racing tickets assigned it:
 * rows[i] went into slots[i].  Each slot must be reserved and each row a distinct
 * non-resident host row (else BAD_INDEX and the pair is skipped).  The row becomes
 * resident with priority clock (fetched this step) and its bytes are copied.
 */
int orc_prefetch_direct(orc_pool *P, const int32_t *slots, const int32_t *rows, int n, int32_t clock)
{
    int status = 0;
    for (int i = 0; i < n; ++i) {
        int32_t s = slots[i], h = rows[i];
        if (s < 0 || s >= P->n_g || P->GPUTokenFree[s] || P->GPUTokenPriority[s] != ORC_RESERVED ||
            h < 0 || h >= P->n_h || P->HostTokenToGPU[h] != ORC_INF) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        P->GPUTokenPriority[s] = clock;
        P->GPUTokenToHost[s] = h;
        P->HostTokenToGPU[h] = s;
        copy_row(P, s, P->host_kv + (size_t)h * P->row_elems);
    }
    return status;
}

/*
 * Guaranteed recall (section 4 step list, section 5.2 "Recall").
 *   (i)   map the selected tokens to host rows; keep the first occurrence of each
 *         row in (b, j, i) order;
 *   (ii)  resident rows are hits: their priority is raised to clock (protect);
 *   (iii) M = number of missing rows; evict max(0, M - free) slots (Free);
 *   (iv)  allocate the missing rows, in order (Allocate);
 *   (v)   copy each recalled row host -> GPU pool.  A row the prefetch staged this
 *         step is counted in staged_used; its bytes are the host row's bytes;
 *   (vi)  out_slot[b][j][i] = GPU slot of sel[b][j][i], -1 for padding and for rows
 *         that found no slot.
 * staged_rows[b*stage_stride + i], i < staged_count[b]: host rows the prefetch
 * staged for request b this step (may be NULL).
 * reserve_cap >= 0 selects direct-to-slot mode: the rows listed in staged_rows are
 * the ones this step's prefetch already put into reserved slots (they are hits, and
 * staged_used counts those selected); before (iii) the reserve left unused returns
 * to the free slots, (iii) evicts for the misses plus reserve_cap more slots (as far
 * as evictable slots go: a short reserve is no exhaustion), and after (iv) the
 * reserve_cap lowest-index free slots become the next reserve, listed in
 * reserve_out (count in *reserve_n_out).  reserve_cap < 0: reserved slots are left
 * as they are (neither free nor evictable).
 */
int orc_prefetch_recall(orc_pool *P, const int32_t *sel, const int32_t *req_to_host, int B,
                        int n_q, int k, int L_max, const int32_t *staged_rows,
                        const int32_t *staged_count, int stage_stride, int32_t clock,
                        int32_t *out_slot, orc_stats *st, int reserve_cap, int32_t *reserve_out,
                        int32_t *reserve_n_out)
{
    int status = 0;
    size_t F = (size_t)B * n_q * k;
    uint8_t *seen = (uint8_t *)calloc((size_t)P->n_h, 1);
    int32_t *miss = (int32_t *)malloc(sizeof(int32_t) * (F > 0 ? F : 1));
    int32_t *miss_req = (int32_t *)malloc(sizeof(int32_t) * (F > 0 ? F : 1));
    int n_miss = 0;
    int64_t n_sel = 0, n_unique = 0, n_hits = 0;

    /* direct-to-slot mode: the rows this step's prefetch put into slots (any request) */
    const int direct = reserve_cap >= 0;
    uint8_t *pref = NULL;
    int64_t used_hits = 0;
    if (direct && staged_rows && staged_count) {
        pref = (uint8_t *)calloc((size_t)P->n_h, 1);
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < staged_count[b]; ++t) {
                int32_t h = staged_rows[(size_t)b * stage_stride + t];
                if (h >= 0 && h < P->n_h)
                    pref[h] = 1;
            }
    }

    /* (i) + (ii) */
    for (size_t f = 0; f < F; ++f) {
        int32_t p = sel[f];
        if (p < 0)
            continue;
        int b = (int)(f / ((size_t)n_q * k));
        if (p >= L_max) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        int32_t h = req_to_host[(size_t)b * L_max + p];
        if (h < 0 || h >= P->n_h) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        ++n_sel;
        if (seen[h])
            continue;
        seen[h] = 1;
        ++n_unique;
        int32_t g = P->HostTokenToGPU[h];
        if (g != ORC_INF) {
            ++n_hits;
            P->GPUTokenPriority[g] = clock;
            if (pref && pref[h])
                ++used_hits;  /* a miss the direct prefetch turned into a hit */
        } else {
            miss[n_miss] = h;
            miss_req[n_miss] = b;
            ++n_miss;
        }
    }
    free(seen);
    free(pref);

    /* (iii); in direct-to-slot mode the unused reserve returns to the free slots and
       the evictions also cover the next reserve */
    if (direct)
        orc_reserve_release(P);
    int32_t n_ev = 0;
    int need = n_miss + (direct ? reserve_cap : 0) - P->n_free;
    if (direct) {  /* a short reserve is not an exhaustion: only misses left out are */
        int nc = orc_evictable(P, clock);
        need = need < nc ? need : nc;
    }
    if (need > 0)
        status |= orc_pool_evict(P, need, clock, &n_ev);

    /* (iv) */
    int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_miss > 0 ? n_miss : 1));
    status |= orc_pool_alloc(P, miss, n_miss, clock, NULL, slots);
    if (direct) {
        int nr = orc_reserve_take(P, reserve_cap, reserve_out);
        if (reserve_n_out)
            *reserve_n_out = nr;
    }

    /* (v) */
    int64_t recalled = 0, used = 0, staged_total = 0;
    for (int i = 0; i < n_miss; ++i) {
        if (slots[i] < 0)
            continue;
        ++recalled;
        copy_row(P, slots[i], P->host_kv + (size_t)miss[i] * P->row_elems);
        if (!direct && staged_rows && staged_count) {
            int b = miss_req[i];
            for (int t = 0; t < staged_count[b]; ++t)
                if (staged_rows[(size_t)b * stage_stride + t] == miss[i]) {
                    ++used;
                    break;
                }
        }
    }
    if (staged_count)
        for (int b = 0; b < B; ++b)
            staged_total += staged_count[b];

    /* (vi) */
    for (size_t f = 0; f < F; ++f) {
        int32_t p = sel[f];
        out_slot[f] = -1;
        if (p < 0 || p >= L_max)
            continue;
        int b = (int)(f / ((size_t)n_q * k));
        int32_t h = req_to_host[(size_t)b * L_max + p];
        if (h < 0 || h >= P->n_h)
            continue;
        int32_t g = P->HostTokenToGPU[h];
        out_slot[f] = g == ORC_INF ? -1 : g;
    }

    if (st) {
        st->steps += 1;
        st->selected += n_sel;
        st->unique_rows += n_unique;
        st->hits += n_hits;
        st->misses += n_miss;
        st->recalled += recalled;
        st->unrecalled += n_miss - recalled;
        st->evicted += n_ev;
        st->staged += staged_total;
        st->staged_used += direct ? used_hits : used;
    }
    free(slots);
    free(miss);
    free(miss_req);
    return status;
}

/*
 * Write-through append of the token each request generates (section 2, "offload":
 * KV is backed up to the host when generated, which is why eviction moves no
 * data).  For request b: p = ctx_len[b]; host row h = req_to_host[b][p] gets the new
 * KV; the indexer K cache gets the new k^I row; ctx_len[b] += 1; the new rows get
 * GPU slots (evicting first if the pool is short) with priority clock, and their KV
 * is copied into the GPU pool.
 */
int orc_append(orc_pool *P, uint8_t *k_index, int32_t *ctx_len, const int32_t *req_to_host,
               int B, int L_max, int D, const uint16_t *new_kv, const uint8_t *new_k_index,
               int32_t clock, orc_stats *st)
{
    int status = 0;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    int32_t *src = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    int n = 0;
    for (int b = 0; b < B; ++b) {
        int p = ctx_len[b];
        if (p < 0 || p >= L_max) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        int32_t h = req_to_host[(size_t)b * L_max + p];
        if (h < 0 || h >= P->n_h) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        memcpy(P->host_kv + (size_t)h * P->row_elems, new_kv + (size_t)b * P->row_elems,
               sizeof(uint16_t) * (size_t)P->row_elems);
        memcpy(k_index + ((size_t)b * L_max + p) * D, new_k_index + (size_t)b * D, (size_t)D);
        ctx_len[b] = p + 1;
        /* A new token's row has no GPU copy yet.  One that is already resident, or that
           an earlier request of this call appends too, is written through but takes no
           slot and frees none (flagged). */
        int repeat = 0;
        for (int i = 0; i < n; ++i)
            repeat |= rows[i] == h;
        if (P->HostTokenToGPU[h] != ORC_INF || repeat) {
            status |= ORC_BAD_INDEX;
            continue;
        }
        rows[n] = h;
        src[n] = b;
        ++n;
    }
    int32_t n_ev = 0;
    if (n > P->n_free)
        status |= orc_pool_evict(P, n - P->n_free, clock, &n_ev);
    int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    status |= orc_pool_alloc(P, rows, n, clock, NULL, slots);
    for (int i = 0; i < n; ++i)
        if (slots[i] >= 0)
            copy_row(P, slots[i], new_kv + (size_t)src[i] * P->row_elems);
    if (st) {
        st->appended += n;
        st->evicted += n_ev;
    }
    free(slots);
    free(rows);
    free(src);
    return status;
}

/* ------------------------------------------------------------------------- */
/* Intra-query prefetch (section 6.1)                                         */
/* ------------------------------------------------------------------------- */

/*
 * Tokens of request b that the fused prefetch may stage this step: some query j has
 * score > s_hat[b][j] and the token's host row is not resident.  Listed once each, in
 * ascending token order, into cand[b*L_max + i], i < cand_count[b].  cap[b] is the
 * prefetch bound of request b: min(stage_stride, ceil(ctx_len[b] / cap_div)).
 * The set is what the GPU stages when cand_count[b] <= cap[b]; above the cap the GPU
 * stages some cap[b] of them (the order the counter is taken in decides which).
 */
void orc_prefetch_candidates(const float *scores, const float *s_hat, const int32_t *ctx_len,
                             const int32_t *req_to_host, const int32_t *HostTokenToGPU, int n_h,
                             int B, int n_q, int L_max, int stage_stride, int cap_div,
                             int32_t *cand, int32_t *cand_count, int32_t *cap)
{
    for (int b = 0; b < B; ++b) {
        int n = 0;
        for (int p = 0; p < L_max; ++p) {
            int pass = 0;
            for (int j = 0; j < n_q; ++j) {
                size_t row = (size_t)b * n_q + j;
                if (p < valid_len(ctx_len[b], n_q, j) && scores[row * L_max + p] > s_hat[row])
                    pass = 1;
            }
            if (!pass)
                continue;
            int32_t h = req_to_host[(size_t)b * L_max + p];
            if (h < 0 || h >= n_h || HostTokenToGPU[h] != ORC_INF)
                continue;
            cand[(size_t)b * L_max + n++] = p;
        }
        cand_count[b] = n;
        long c = ((long)ctx_len[b] + cap_div - 1) / cap_div;
        cap[b] = (int32_t)(c < stage_stride ? c : stage_stride);
    }
}

/* ------------------------------------------------------------------------- */
/* Inter-query prefetch (section 6.2)                                         */
/* ------------------------------------------------------------------------- */

/* order-preserving 32-bit key of an fp32 value (a larger value has a larger key;
   -0 is folded onto +0) */
static uint32_t orc_order_key(float x)
{
    if (x == 0.0f)
        x = 0.0f;
    uint32_t u;
    memcpy(&u, &x, sizeof(u));
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

/*
 * Approximate top-k of one query's scores (section 6.2): each score is shifted by the
 * predicted k-th score, x = s - s_hat (fp32), and binned by the top 8 bits of x's
 * order-preserving key into S_0 .. S_255 (S_255 holds the largest values).  The top j
 * bins are taken, j the largest with S_{256-j} + ... + S_255 <= k; bin 255 - j is the
 * threshold bin (-1 when every bin fits).  Returns the threshold bin; hist receives
 * S_0 .. S_255 and *subset_n the count of the taken bins, which by construction obeys
 * the section's inequality k - S_{255-j} < subset_n <= k (when the threshold bin exists).
 */
int orc_approx_topk_bins(const float *scores, int L, float s_hat, int k, int32_t *hist, int32_t *subset_n)
{
    for (int i = 0; i < 256; ++i)
        hist[i] = 0;
    for (int p = 0; p < L; ++p) {
        float x = scores[p] - s_hat;
        hist[orc_order_key(x) >> 24] += 1;
    }
    int64_t sum = 0;
    int bin = 255;
    while (bin >= 0 && sum + hist[bin] <= k) {
        sum += hist[bin];
        --bin;
    }
    *subset_n = (int32_t)sum;
    return bin;
}

/*
 * Prefill chunk (section 6.2 with the prefill kernel of section 6.3): request b scores
 * its last C tokens as queries (query i sees valid_len(ctx_len[b], C, i) keys, as in
 * orc_indexer_score with n_q = C).  Queries are taken in blocks of qb; when a block is
 * scored, its prefetch candidates are the tokens that some query of the block puts
 * above its threshold bin (the approximate top-k above, shift s_hat[b]) and whose host
 * row is not resident, in ascending token order, once per block.
 *   thr_bin, subset_n [B][C]; cand [B][n_blocks][L_max], cand_count [B][n_blocks],
 *   n_blocks = ceil(C / qb).
 */
void orc_prefill_candidates(const float *scores, const float *s_hat, const int32_t *ctx_len, int B, int C,
                            int L_max, int k, int qb, const int32_t *req_to_host,
                            const int32_t *HostTokenToGPU, int n_h, int32_t *thr_bin, int32_t *subset_n,
                            int32_t *cand, int32_t *cand_count)
{
    int32_t hist[256];
    const int nb = (C + qb - 1) / qb;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < C; ++i) {
            size_t row = (size_t)b * C + i;
            int L = valid_len(ctx_len[b], C, i);
            thr_bin[row] = orc_approx_topk_bins(scores + row * L_max, L, s_hat[b], k, hist, &subset_n[row]);
        }
        for (int blk = 0; blk < nb; ++blk) {
            int n = 0;
            int32_t *out = cand + ((size_t)b * nb + blk) * L_max;
            for (int p = 0; p < L_max; ++p) {
                int pass = 0;
                for (int i = blk * qb; i < C && i < (blk + 1) * qb; ++i) {
                    size_t row = (size_t)b * C + i;
                    if (p >= valid_len(ctx_len[b], C, i))
                        continue;
                    float x = scores[row * L_max + p] - s_hat[b];
                    if ((int)(orc_order_key(x) >> 24) > thr_bin[row])
                        pass = 1;
                }
                if (!pass)
                    continue;
                int32_t h = req_to_host[(size_t)b * L_max + p];
                if (h < 0 || h >= n_h || HostTokenToGPU[h] != ORC_INF)
                    continue;
                out[n++] = p;
            }
            cand_count[(size_t)b * nb + blk] = n;
        }
    }
}

/* s_hat <- alpha s_hat + (1 - alpha) kth, in fp32; the first finite observation
   replaces the +inf start value; a non-finite kth (empty context) is skipped */
void orc_ema_update(float *s_hat, const float *kth, int n, float alpha)
{
    for (int i = 0; i < n; ++i) {
        float x = kth[i];
        if (!isfinite(x))
            continue;
        if (isinf(s_hat[i]) && s_hat[i] > 0) {
            s_hat[i] = x;
            continue;
        }
        float a = alpha * s_hat[i];
        float c = (1.0f - alpha) * x;
        s_hat[i] = a + c;
    }
}

/* ------------------------------------------------------------------------- */
/* Sparse MLA decode over the selected rows (section 2, MLA; section 3.2)     */
/* ------------------------------------------------------------------------- */

/* bf16 bits -> double (exact) */
static double orc_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof(f));
    return (double)f;
}

/*
 * Attention of query token (b, j) over its selected latent rows (MLA with the key
 * and value up-projections absorbed into the query and the output: every head reads
 * the same d_c + rope latent row).  For head h:
 *   s_i = scale * sum_{d < dqk} q[b][j][h][d] * kv[slot_i][d]     (dqk = 576)
 *   o[d] = sum_i softmax(s)_i * kv[slot_i][d]                      (d < dv = 512)
 *   lse = log(sum_i exp(s_i))
 * over the selected entries i < k whose slot (out_slot[b][j][i]) is >= 0; a row with
 * no such entry gives o = 0 and lse = -inf.  Everything in fp64 from the bf16 inputs.
 *   q [B][n_q][H][dqk] bf16; kv [n_g][row] bf16; out_slot [B][n_q][k];
 *   o [B][n_q][H][dv] double; lse [B][n_q][H] double.
 */
void orc_sparse_mla_decode(const uint16_t *q, const uint16_t *kv, int row, const int32_t *out_slot, int B,
                           int n_q, int H, int dqk, int dv, int k, int n_g, double scale, double *o, double *lse)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    for (int b = 0; b < B; ++b)
        for (int j = 0; j < n_q; ++j)
            for (int h = 0; h < H; ++h) {
                const uint16_t *qh = q + (((size_t)b * n_q + j) * H + h) * dqk;
                const int32_t *sl = out_slot + ((size_t)b * n_q + j) * k;
                double *oh = o + (((size_t)b * n_q + j) * H + h) * dv;
                double m = -INFINITY;
                for (int i = 0; i < k; ++i) {
                    s[i] = -INFINITY;
                    if (sl[i] < 0 || sl[i] >= n_g)
                        continue;
                    const uint16_t *r = kv + (size_t)sl[i] * row;
                    double acc = 0.0;
                    for (int d = 0; d < dqk; ++d)
                        acc += orc_bf16(qh[d]) * orc_bf16(r[d]);
                    s[i] = scale * acc;
                    if (s[i] > m)
                        m = s[i];
                }
                for (int d = 0; d < dv; ++d)
                    oh[d] = 0.0;
                double l = 0.0;
                if (m != -INFINITY) {
                    for (int i = 0; i < k; ++i) {
                        if (s[i] == -INFINITY)
                            continue;
                        double p = exp(s[i] - m);
                        l += p;
                        const uint16_t *r = kv + (size_t)sl[i] * row;
                        for (int d = 0; d < dv; ++d)
                            oh[d] += p * orc_bf16(r[d]);
                    }
                    for (int d = 0; d < dv; ++d)
                        oh[d] /= l;
                }
                lse[((size_t)b * n_q + j) * H + h] = m == -INFINITY ? -INFINITY : m + log(l);
            }
    free(s);
}

/* storage law of the five metadata arrays (section 5.1): 4 N_H + 13 N_G bytes */
int64_t orc_metadata_bytes(int64_t n_h, int64_t n_g)
{
    return (int64_t)sizeof(int32_t) * n_h                          /* HostTokenToGPU   */
           + (int64_t)(sizeof(uint8_t) + 3 * sizeof(int32_t)) * n_g; /* free + 3 slot arrays */
}
