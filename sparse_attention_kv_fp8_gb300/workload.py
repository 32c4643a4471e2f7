"""Seeded synthetic inputs for the ECHO decode step.

This module is the one piece shared by the CUDA path's callers (tests, bench)
and the CPU oracle: it makes input bytes and nothing else.  It holds none of
the step's arithmetic (no scoring, no selection, no cache-manager rule); it only
draws random numbers and encodes them into the storage formats the step reads
(FP8 e4m3 for the lightning-indexer q/k, fp32 head weights, bf16 latent KV).

Workload shapes follow the ECHO review (marsggbo.github.io, "OSDI'26 | ECHO"):
DeepSeek-V3.2 indexer with H_index = 64 heads and d_index = 128 (section 2,
"DSA indexer"), latent KV of d_c = 512 plus 64 rope dims per token (section 2,
"MLA"), a per-model host pool and a per-layer GPU pool (section 4 and
section 5.1).  The real workloads (InfiniteBench, ShareGPT) are not used; these
seeded draws stand in for them.

Random numbers come from numpy's PCG64 seeded through a SeedSequence of
(seed, stream), which gives the same bytes on x86 and Arm for a given numpy.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

H_INDEX = 64          # indexer heads
D_INDEX = 128         # indexer head dim (bytes per k^I row in e4m3)
KV_ELEMS = 576        # latent KV per token: 512 (d_c) + 64 rope, bf16
KV_BYTES = KV_ELEMS * 2
INF_I32 = 2**31 - 1   # the "empty" sentinel of the residency maps

# stream ids, so that every array has its own independent draw
_S_Q, _S_W, _S_K, _S_KV, _S_POOL, _S_EPS, _S_NEWKV, _S_NEWK, _S_MLAQ, _S_BKV, _S_BSC = range(1, 12)


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), int(stream)])))


# ---------------------------------------------------------------------------
# storage encodings (input formats, not the method)
# ---------------------------------------------------------------------------

def e4m3_encode_direct(x: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3fn code (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits; subnormal step 2^-9; largest finite 448), ties to even, saturating at +-448.
    The input is first rounded to float32 (the draws are float32 or float64)."""
    xf = np.asarray(x, dtype=np.float32)
    a = np.minimum(np.abs(xf), np.float32(448.0))
    u = a.view(np.uint32)
    # normal range: round the 23-bit float32 mantissa to 3 bits, half to even
    r = u + np.uint32(0x7FFFF) + ((u >> np.uint32(20)) & np.uint32(1))
    e = (r >> np.uint32(23)).astype(np.int32) - 127 + 7
    code = (e << 3) | ((r >> np.uint32(20)) & np.uint32(7)).astype(np.int32)
    # subnormal range (|x| < 2^-6): code = round(|x| / 2^-9); code 8 is the smallest normal
    sub = a < np.float32(2.0 ** -6)
    code = np.where(sub, np.rint(a * np.float32(512.0)).astype(np.int32), code)
    sign = np.where(np.signbit(xf), 0x80, 0)
    return (code | sign).astype(np.uint8)


_E4M3_TABLE = None


def _e4m3_table() -> np.ndarray:
    """The code of every float32 class (top 16 bits, whether any of the low 16 bits is
    set), from the direct encoder.  The rounding decision reads the round bit (bit 19
    or higher) and whether any lower bit is set, so the class decides the code."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
        reps = np.stack([hi, hi | np.uint32(1)], axis=1).reshape(-1)
        with np.errstate(invalid="ignore"):
            _E4M3_TABLE = e4m3_encode_direct(reps.view(np.float32))
    return _E4M3_TABLE


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """e4m3_encode_direct through a 128K-entry table (same codes for finite inputs)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    idx = ((u >> np.uint32(16)) << np.uint32(1)) | ((u & np.uint32(0xFFFF)) != 0).astype(np.uint32)
    return _e4m3_table()[idx]


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern (uint16), round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def fp8_normal(g: np.ndarray | np.random.Generator, shape, clamp: float = 8.0) -> np.ndarray:
    """N(0,1) draws clamped to [-clamp, clamp], encoded e4m3 (|x| <= 8 per the workload)."""
    x = g.standard_normal(size=shape, dtype=np.float32) if isinstance(g, np.random.Generator) else g
    return e4m3_encode(np.clip(x, -clamp, clamp))


# ---------------------------------------------------------------------------
# indexer inputs
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class IndexerInputs:
    q: np.ndarray        # uint8  [B][n_q][H][D]   e4m3 codes
    w: np.ndarray        # f32    [B][n_q][H]
    k_index: np.ndarray  # uint8  [B][L_max][D]    e4m3 codes
    ctx_len: np.ndarray  # int32  [B]
    q_float: np.ndarray  # f64    [B][n_q][H][D]   pre-rounding draw (for correlated steps)


def indexer_inputs(B: int, n_q: int, L_max: int, ctx_len, seed: int,
                   H: int = H_INDEX, D: int = D_INDEX, chunk_rows: int = 1 << 18) -> IndexerInputs:
    ctx = np.broadcast_to(np.asarray(ctx_len, dtype=np.int32), (B,)).copy()
    if np.any(ctx < 0) or np.any(ctx > L_max):
        raise ValueError("ctx_len out of range")
    gq = rng(seed, _S_Q)
    qf = np.clip(gq.standard_normal(size=(B, n_q, H, D)), -8.0, 8.0)
    q = e4m3_encode(qf)
    w = rng(seed, _S_W).random(size=(B, n_q, H), dtype=np.float64).astype(np.float32)
    gk = rng(seed, _S_K)
    k = np.empty((B * L_max, D), dtype=np.uint8)
    for r0 in range(0, B * L_max, chunk_rows):
        r1 = min(B * L_max, r0 + chunk_rows)
        k[r0:r1] = fp8_normal(gk, (r1 - r0, D))
    return IndexerInputs(q=q, w=w, k_index=k.reshape(B, L_max, D), ctx_len=ctx, q_float=qf)


def next_query(q_float: np.ndarray, rho: float, seed: int, step: int):
    """One step of q_{t+1} = rho*q_t + sqrt(1-rho^2)*eps (eps ~ N(0,1)), clamped and encoded.

    The step-to-step correlation of the indexer query sets how much consecutive
    top-k sets overlap, which in turn sets the GPU-pool hit rate.
    Returns (q_float_next, q_e4m3_next)."""
    eps = rng(seed * 1000003 + step, _S_EPS).standard_normal(size=q_float.shape)
    qn = np.clip(rho * q_float + math.sqrt(max(0.0, 1.0 - rho * rho)) * eps, -8.0, 8.0)
    return qn, e4m3_encode(qn)


# ---------------------------------------------------------------------------
# latent KV pools
# ---------------------------------------------------------------------------

def host_kv_pool(n_h: int, seed: int, n_random: int | None = None, out: np.ndarray | None = None,
                 chunk_rows: int = 1 << 16) -> np.ndarray:
    """Host pool [n_h][576] bf16 bits.  Rows < n_random hold N(0,1) draws; the rest
    (rows no request of the workload references) hold a cheap per-row pattern so
    that every row is still distinct."""
    if n_random is None:
        n_random = n_h
    if out is None:
        out = np.empty((n_h, KV_ELEMS), dtype=np.uint16)
    g = rng(seed, _S_KV)
    for r0 in range(0, n_random, chunk_rows):
        r1 = min(n_random, r0 + chunk_rows)
        out[r0:r1] = bf16_encode(g.standard_normal(size=(r1 - r0, KV_ELEMS), dtype=np.float32))
    if n_random < n_h:
        rows = np.arange(n_random, n_h, dtype=np.uint32)
        col = np.arange(KV_ELEMS, dtype=np.uint32)
        for r0 in range(0, rows.size, chunk_rows):
            rr = rows[r0:r0 + chunk_rows, None]
            out[n_random + r0:n_random + r0 + rr.shape[0]] = ((rr * np.uint32(2654435761) + col) & np.uint32(0x3FFF)).astype(np.uint16)
    return out


def new_tokens(B: int, seed: int, step: int):
    """KV row (bf16 bits) and k^I row (e4m3) of the token each request appends at `step`."""
    kv = bf16_encode(rng(seed * 1000003 + step, _S_NEWKV).standard_normal(size=(B, KV_ELEMS), dtype=np.float32))
    kI = fp8_normal(rng(seed * 1000003 + step, _S_NEWK), (B, D_INDEX))
    return kv, kI


def mla_queries(B: int, n_q: int, seed: int, heads: int = 128) -> np.ndarray:
    """Absorbed MLA queries [B][n_q][heads][576] bf16 bits, N(0,1) draws (section 2: the
    attention has 128 heads over the 512 + 64 latent row)."""
    g = rng(seed, _S_MLAQ)
    return bf16_encode(g.standard_normal(size=(B, n_q, heads, KV_ELEMS), dtype=np.float32))


# ---------------------------------------------------------------------------
# block-level / GQA variant of the cache manager (the review's section 8: the cache
# manager carries over to block-sparse attention with coarser metadata and a KV-head
# dimension).  A pool row is one block of `block` tokens of one KV head, K and V of
# head_dim each in bf16; a selection row is one (request, KV head) pair.  The shapes
# of a GQA model with 8 KV heads of 128 dims and an NSA-style choice of 16 blocks of
# 64 tokens stand in for a real model.
# ---------------------------------------------------------------------------
GQA_KV_HEADS, GQA_HEAD_DIM, GQA_BLOCK, GQA_TOPK_BLOCKS = 8, 128, 64, 16


def block_row_elems(block: int = GQA_BLOCK, head_dim: int = GQA_HEAD_DIM) -> int:
    """bf16 elements of one block row: K and V of `block` tokens of one KV head."""
    return 2 * block * head_dim


def block_kv_pool(n_units: int, row_elems: int, seed: int, out: np.ndarray | None = None,
                  chunk_rows: int = 4096) -> np.ndarray:
    """Host pool of block rows [n_units][row_elems] bf16 bits, N(0,1) draws."""
    out = np.empty((n_units, row_elems), np.uint16) if out is None else out
    g = rng(seed, _S_BKV)
    for r0 in range(0, n_units, chunk_rows):
        r1 = min(n_units, r0 + chunk_rows)
        out[r0:r1] = bf16_encode(g.standard_normal((r1 - r0, row_elems), dtype=np.float32))
    return out


def block_scores(rows: int, n_blocks: int, seed: int, steps: int, rho: float) -> list[np.ndarray]:
    """Scores of every block for `steps` consecutive decode steps, [rows][1][n_blocks]
    fp32 each; step t+1 = rho * step t + sqrt(1 - rho^2) * fresh N(0,1), so that the
    top blocks of consecutive steps overlap (rho = 0: independent steps)."""
    g = rng(seed, _S_BSC)
    s = g.standard_normal((rows, 1, n_blocks), dtype=np.float32)
    out = [s.copy()]
    c = np.float32(math.sqrt(max(0.0, 1.0 - rho * rho)))
    for _ in range(steps - 1):
        s = np.float32(rho) * s + c * g.standard_normal((rows, 1, n_blocks), dtype=np.float32)
        out.append(s.astype(np.float32))
    return out


def req_to_host(B: int, L_max: int, base: int = 0) -> np.ndarray:
    """Host row of token p of request b: base + b*L_max + p (each request owns a contiguous range)."""
    return (base + np.arange(B, dtype=np.int64)[:, None] * L_max + np.arange(L_max, dtype=np.int64)[None, :]).astype(np.int32)


@dataclasses.dataclass
class PoolState:
    """Initial GPU-pool metadata (the five fixed-length arrays) plus counters."""
    n_g: int
    n_h: int
    gpu_token_free: np.ndarray       # uint8 [n_g]   1 = free
    gpu_token_priority: np.ndarray   # int32 [n_g]   -1 when free
    gpu_indices_buffer: np.ndarray   # int32 [n_g]   -1 = invalid
    gpu_token_to_host: np.ndarray    # int32 [n_g]   INF when empty
    host_token_to_gpu: np.ndarray    # int32 [n_h]   INF when not resident
    n_free: int
    idx_count: int


def empty_pool(n_g: int, n_h: int) -> PoolState:
    return PoolState(n_g, n_h,
                     np.ones(n_g, np.uint8), np.full(n_g, -1, np.int32), np.full(n_g, -1, np.int32),
                     np.full(n_g, INF_I32, np.int32), np.full(n_h, INF_I32, np.int32), n_g, 0)


def resident_pool(n_g: int, n_h: int, resident_rows: np.ndarray, clocks: np.ndarray, seed: int,
                  scatter: bool = True) -> PoolState:
    """Pool holding `resident_rows` (distinct host rows) with the given priorities.
    Slots are drawn at random (scatter=True) or packed from slot 0."""
    resident_rows = np.asarray(resident_rows, dtype=np.int64)
    n = resident_rows.size
    if n > n_g or np.unique(resident_rows).size != n:
        raise ValueError("resident rows must be distinct and fit in the pool")
    st = empty_pool(n_g, n_h)
    slots = rng(seed, _S_POOL).permutation(n_g)[:n] if scatter else np.arange(n)
    st.gpu_token_free[slots] = 0
    st.gpu_token_priority[slots] = np.asarray(clocks, dtype=np.int32)
    st.gpu_token_to_host[slots] = resident_rows.astype(np.int32)
    st.host_token_to_gpu[resident_rows] = slots.astype(np.int32)
    st.n_free = n_g - n
    return st


def random_resident_rows(candidates: int, n: int, seed: int, stream_off: int = 0) -> np.ndarray:
    """n distinct host rows drawn uniformly from [0, candidates)."""
    g = rng(seed, _S_POOL + 100 + stream_off)
    return np.sort(g.choice(candidates, size=n, replace=False)).astype(np.int64)


def random_clocks(n: int, t: int, seed: int) -> np.ndarray:
    """Priorities U{0..t-1} for pre-resident rows (older than the step clock t)."""
    return rng(seed, _S_POOL + 200).integers(0, t, size=n).astype(np.int32)
