"""CPU oracle of the ECHO decode step (ctypes wrapper around echo_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only tests/, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  The product path (the CUDA
library and its Python binding) never imports, links or runs anything here.

Every function follows the ECHO review page (marsggbo.github.io, "OSDI'26 |
ECHO"); the C source cites the section behind each step.  Parity status: every
function is pinned by tests/test_oracle_pins.py (closed forms, brute force, the
page's worked allocation example, and the lossless / byte-equality invariants).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "echo_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, f"libecho_oracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None

INF = 2**31 - 1
POOL_EXHAUSTED, BAD_INDEX, PREFETCH_CAP_HIT = 1, 2, 8
RESERVED = -2   # priority of a slot set aside for the direct-to-slot prefetch


def build(force: bool = False) -> str:
    """Compile echo_oracle.c with gcc (single-threaded, strict fp: no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Pool(ctypes.Structure):
    _fields_ = [("n_g", ctypes.c_int32), ("n_h", ctypes.c_int32), ("row_elems", ctypes.c_int32),
                ("GPUTokenFree", ctypes.c_void_p), ("GPUTokenPriority", ctypes.c_void_p),
                ("GPUIndicesBuffer", ctypes.c_void_p), ("GPUTokenToHost", ctypes.c_void_p),
                ("HostTokenToGPU", ctypes.c_void_p), ("gpu_kv", ctypes.c_void_p),
                ("host_kv", ctypes.c_void_p), ("n_free", ctypes.c_int32), ("idx_count", ctypes.c_int32)]


STAT_FIELDS = ("steps", "selected", "unique_rows", "hits", "misses", "recalled", "unrecalled",
               "evicted", "staged", "staged_used", "appended")


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in STAT_FIELDS]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n in STAT_FIELDS}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_value.restype = ctypes.c_double
            L.orc_indexer_score_one.argtypes = [P, P, P, I, I, I, I, I, I, I]
            L.orc_indexer_score_one.restype = F
            L.orc_indexer_score.argtypes = [P, P, P, P, I, I, I, I, I, P]
            L.orc_indexer_score.restype = None
            L.orc_select_topk.argtypes = [P, P, I, I, I, I, P, P]
            L.orc_select_topk.restype = None
            L.orc_pool_init.argtypes = [P]
            L.orc_pool_init.restype = None
            L.orc_pool_alloc.argtypes = [P, P, I, ctypes.c_int32, P, P]
            L.orc_pool_alloc.restype = I
            L.orc_pool_evict.argtypes = [P, I, ctypes.c_int32, P]
            L.orc_pool_evict.restype = I
            L.orc_prefetch_recall.argtypes = [P, P, P, I, I, I, I, P, P, I, ctypes.c_int32, P, P, I, P, P]
            L.orc_prefetch_recall.restype = I
            L.orc_append.argtypes = [P, P, P, P, I, I, I, P, P, ctypes.c_int32, P]
            L.orc_prefetch_direct.argtypes = [P, P, P, I, ctypes.c_int32]
            L.orc_prefetch_direct.restype = I
            L.orc_append.restype = I
            L.orc_prefetch_candidates.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P, P]
            L.orc_prefetch_candidates.restype = None
            L.orc_approx_topk_bins.argtypes = [P, I, F, I, P, P]
            L.orc_approx_topk_bins.restype = I
            L.orc_prefill_candidates.argtypes = [P, P, P, I, I, I, I, I, P, P, I, P, P, P, P]
            L.orc_prefill_candidates.restype = None
            L.orc_sparse_mla_decode.argtypes = [P, P, I, P, I, I, I, I, I, I, I, ctypes.c_double, P, P]
            L.orc_sparse_mla_decode.restype = None
            L.orc_ema_update.argtypes = [P, P, I, F]
            L.orc_ema_update.restype = None
            L.orc_metadata_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.orc_metadata_bytes.restype = ctypes.c_int64
            _lib = L
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _arr(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# indexer / top-k / EMA
# ---------------------------------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(int(code))


def indexer_score(q, w, k_index, ctx_len, out: np.ndarray | None = None) -> np.ndarray:
    """scores [B][n_q][L_max] f32; entries past each query's visible length are NaN."""
    q = _arr(q, np.uint8)
    w = _arr(w, np.float32)
    k_index = _arr(k_index, np.uint8)
    ctx_len = _arr(ctx_len, np.int32)
    B, n_q, H, D = q.shape
    L_max = k_index.shape[1]
    assert k_index.shape == (B, L_max, D) and w.shape == (B, n_q, H)
    if out is None:
        out = np.full((B, n_q, L_max), np.nan, dtype=np.float32)
    lib().orc_indexer_score(_p(q), _p(w), _p(k_index), _p(ctx_len), B, n_q, L_max, H, D, _p(out))
    return out


def indexer_score_one(q, w, k_index, b: int, j: int, p: int) -> float:
    q = _arr(q, np.uint8)
    w = _arr(w, np.float32)
    k_index = _arr(k_index, np.uint8)
    B, n_q, H, D = q.shape
    return lib().orc_indexer_score_one(_p(q), _p(w), _p(k_index), n_q, k_index.shape[1], H, D, b, j, p)


def select_topk(scores, ctx_len, k: int):
    scores = _arr(scores, np.float32)
    ctx_len = _arr(ctx_len, np.int32)
    B, n_q, L_max = scores.shape
    sel = np.empty((B, n_q, k), np.int32)
    kth = np.empty((B, n_q), np.float32)
    lib().orc_select_topk(_p(scores), _p(ctx_len), B, n_q, L_max, k, _p(sel), _p(kth))
    return sel, kth


def ema_update(s_hat, kth, alpha: float = 0.5) -> np.ndarray:
    s = np.array(s_hat, dtype=np.float32, copy=True).ravel()
    kth = _arr(kth, np.float32).ravel()
    lib().orc_ema_update(_p(s), _p(kth), s.size, float(alpha))
    return s.reshape(np.shape(s_hat))


def metadata_bytes(n_h: int, n_g: int) -> int:
    return int(lib().orc_metadata_bytes(n_h, n_g))


def prefetch_candidates(scores, s_hat, ctx_len, req_to_host, host_token_to_gpu, stage_stride: int,
                        cap_div: int):
    """Per request: (sorted candidate token list, cap)."""
    scores = _arr(scores, np.float32)
    s_hat = _arr(s_hat, np.float32)
    ctx_len = _arr(ctx_len, np.int32)
    req_to_host = _arr(req_to_host, np.int32)
    h2g = _arr(host_token_to_gpu, np.int32)
    B, n_q, L_max = scores.shape
    cand = np.empty((B, L_max), np.int32)
    cnt = np.empty(B, np.int32)
    cap = np.empty(B, np.int32)
    lib().orc_prefetch_candidates(_p(scores), _p(s_hat), _p(ctx_len), _p(req_to_host), _p(h2g),
                                  h2g.size, B, n_q, L_max, stage_stride, cap_div,
                                  _p(cand), _p(cnt), _p(cap))
    return [cand[b, :cnt[b]].copy() for b in range(B)], cap


def approx_topk_bins(scores_row, s_hat: float, k: int):
    """Approximate top-k of one query's scores (section 6.2): (threshold bin, 256-bin
    histogram of the shifted scores, size of the subset above the threshold bin)."""
    row = _arr(scores_row, np.float32)
    hist = np.zeros(256, np.int32)
    n = np.zeros(1, np.int32)
    t = lib().orc_approx_topk_bins(_p(row), row.size, float(np.float32(s_hat)), int(k), _p(hist), _p(n))
    return int(t), hist, int(n[0])


def prefill_candidates(scores, s_hat, ctx_len, k: int, qb: int, req_to_host, host_token_to_gpu):
    """Prefill chunk of C = scores.shape[1] query tokens per request (section 6.2):
    per query the threshold bin and subset size; per (request, query block) the
    prefetch candidates (tokens some query of the block puts above its threshold bin,
    host row not resident), ascending.  Returns (thr_bin [B][C], subset_n [B][C],
    list over requests of lists over blocks of token arrays)."""
    scores = _arr(scores, np.float32)
    s_hat = _arr(s_hat, np.float32).reshape(-1)
    ctx_len = _arr(ctx_len, np.int32)
    req_to_host = _arr(req_to_host, np.int32)
    h2g = _arr(host_token_to_gpu, np.int32)
    B, C, L_max = scores.shape
    nb = (C + qb - 1) // qb
    thr = np.empty((B, C), np.int32)
    sub = np.empty((B, C), np.int32)
    cand = np.empty((B, nb, L_max), np.int32)
    cnt = np.empty((B, nb), np.int32)
    lib().orc_prefill_candidates(_p(scores), _p(s_hat), _p(ctx_len), B, C, L_max, int(k), int(qb),
                                 _p(req_to_host), _p(h2g), h2g.size, _p(thr), _p(sub), _p(cand), _p(cnt))
    return thr, sub, [[cand[b, i, :cnt[b, i]].copy() for i in range(nb)] for b in range(B)]


def sparse_mla_decode(q, gpu_kv, out_slot, scale: float, dv: int = 512):
    """Attention of each query token's heads over its selected latent rows (fp64):
    q [B][n_q][H][dqk] bf16 bits (uint16), gpu_kv [n_g][row] bf16 bits, out_slot
    [B][n_q][k] (-1 = skipped).  Returns (o [B][n_q][H][dv], lse [B][n_q][H]) float64."""
    q = _arr(q, np.uint16)
    kv = _arr(gpu_kv, np.uint16)
    sl = _arr(out_slot, np.int32)
    B, n_q, H, dqk = q.shape
    k = sl.shape[2]
    o = np.empty((B, n_q, H, dv), np.float64)
    lse = np.empty((B, n_q, H), np.float64)
    lib().orc_sparse_mla_decode(_p(q), _p(kv), kv.shape[1], _p(sl), B, n_q, H, dqk, dv, k, kv.shape[0],
                                float(scale), _p(o), _p(lse))
    return o, lse


# ---------------------------------------------------------------------------
# cache manager
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Pool:
    """The oracle's own copy of one layer's GPU pool plus the (shared) host pool."""
    GPUTokenFree: np.ndarray
    GPUTokenPriority: np.ndarray
    GPUIndicesBuffer: np.ndarray
    GPUTokenToHost: np.ndarray
    HostTokenToGPU: np.ndarray
    gpu_kv: np.ndarray
    host_kv: np.ndarray
    n_free: int
    idx_count: int

    @property
    def n_g(self):
        return self.GPUTokenFree.size

    @property
    def n_h(self):
        return self.HostTokenToGPU.size

    @classmethod
    def empty(cls, n_g: int, n_h: int, host_kv: np.ndarray, row_elems: int = 576):
        P = cls(np.empty(n_g, np.uint8), np.empty(n_g, np.int32), np.empty(n_g, np.int32),
                np.empty(n_g, np.int32), np.empty(n_h, np.int32),
                np.zeros((n_g, row_elems), np.uint16), host_kv, 0, 0)
        with P._c() as c:
            lib().orc_pool_init(ctypes.byref(c))
        return P

    @classmethod
    def from_state(cls, st, host_kv: np.ndarray, gpu_kv: np.ndarray | None = None):
        """From a workload.PoolState; gpu_kv defaults to the host rows of the resident slots."""
        if gpu_kv is None:
            gpu_kv = np.zeros((st.n_g, host_kv.shape[1]), np.uint16)
            occ = np.nonzero(st.gpu_token_free == 0)[0]
            gpu_kv[occ] = host_kv[st.gpu_token_to_host[occ]]
        return cls(st.gpu_token_free.copy(), st.gpu_token_priority.copy(), st.gpu_indices_buffer.copy(),
                   st.gpu_token_to_host.copy(), st.host_token_to_gpu.copy(), gpu_kv, host_kv,
                   int(st.n_free), int(st.idx_count))

    class _Ctx:
        def __init__(self, P):
            self.P = P

        def __enter__(self):
            P = self.P
            for name in ("GPUTokenFree", "GPUTokenPriority", "GPUIndicesBuffer", "GPUTokenToHost",
                         "HostTokenToGPU", "gpu_kv", "host_kv"):
                assert getattr(P, name).flags["C_CONTIGUOUS"], name
            self.c = _Pool(P.n_g, P.n_h, P.gpu_kv.shape[1] if P.gpu_kv.ndim == 2 else 576,
                           _p(P.GPUTokenFree), _p(P.GPUTokenPriority), _p(P.GPUIndicesBuffer),
                           _p(P.GPUTokenToHost), _p(P.HostTokenToGPU), _p(P.gpu_kv), _p(P.host_kv),
                           P.n_free, P.idx_count)
            return self.c

        def __exit__(self, *exc):
            self.P.n_free = int(self.c.n_free)
            self.P.idx_count = int(self.c.idx_count)
            return False

    def _c(self):
        return Pool._Ctx(self)

    def alloc(self, host_idx, clock: int, tickets=None):
        host_idx = _arr(host_idx, np.int32)
        out = np.empty(host_idx.size, np.int32)
        t = None if tickets is None else _arr(tickets, np.int32)
        if t is not None:
            assert t.size == self.n_g
        with self._c() as c:
            status = lib().orc_pool_alloc(ctypes.byref(c), _p(host_idx), host_idx.size, int(clock), _p(t), _p(out))
        return out, status

    def evict(self, n_needed: int, clock: int):
        n = np.zeros(1, np.int32)
        with self._c() as c:
            status = lib().orc_pool_evict(ctypes.byref(c), int(n_needed), int(clock), _p(n))
        return int(n[0]), status

    def prefetch_recall(self, sel, req_to_host, clock: int, staged=None, stats: Stats | None = None,
                        reserve_cap: int = -1):
        """staged: list (per request) of host rows the prefetch staged, or None.  With
        reserve_cap >= 0 (direct-to-slot mode) `staged` lists the rows the prefetch put
        into reserved slots, and the call returns (out_slot, status, next reserve)."""
        sel = _arr(sel, np.int32)
        req_to_host = _arr(req_to_host, np.int32)
        B, n_q, k = sel.shape
        L_max = req_to_host.shape[1]
        out = np.empty_like(sel)
        srows = scnt = None
        stride = 1
        if staged is not None:
            stride = max(1, max((len(x) for x in staged), default=1))
            srows = np.full((B, stride), -1, np.int32)
            scnt = np.zeros(B, np.int32)
            for b, rows in enumerate(staged):
                srows[b, :len(rows)] = rows
                scnt[b] = len(rows)
        st = stats if stats is not None else Stats()
        res = np.full(max(reserve_cap, 1), -1, np.int32)
        res_n = np.zeros(1, np.int32)
        with self._c() as c:
            status = lib().orc_prefetch_recall(ctypes.byref(c), _p(sel), _p(req_to_host), B, n_q, k, L_max,
                                               _p(srows), _p(scnt), stride, int(clock), _p(out),
                                               ctypes.byref(st), int(reserve_cap), _p(res), _p(res_n))
        if reserve_cap >= 0:
            return out, status, res[:int(res_n[0])].copy()
        return out, status

    def append(self, k_index: np.ndarray, ctx_len: np.ndarray, req_to_host, new_kv, new_k_index,
               clock: int, stats: Stats | None = None):
        """In place on k_index, ctx_len and the host pool (write-through).  Reserved
        slots (direct-to-slot prefetch) are left as they are."""
        req_to_host = _arr(req_to_host, np.int32)
        new_kv = _arr(new_kv, np.uint16)
        new_k_index = _arr(new_k_index, np.uint8)
        B, L_max, D = k_index.shape
        st = stats if stats is not None else Stats()
        with self._c() as c:
            status = lib().orc_append(ctypes.byref(c), _p(k_index), _p(ctx_len), _p(req_to_host), B, L_max, D,
                                      _p(new_kv), _p(new_k_index), int(clock), ctypes.byref(st))
        return status

    def prefetch_direct(self, slots, rows, clock: int):
        """The direct-to-slot prefetch of one step as the GPU assigned it: rows[i] went
        into reserved slot slots[i].  Returns the status (BAD_INDEX for invalid pairs)."""
        slots = _arr(slots, np.int32)
        rows = _arr(rows, np.int32)
        assert slots.shape == rows.shape
        with self._c() as c:
            return lib().orc_prefetch_direct(ctypes.byref(c), _p(slots), _p(rows), slots.size, int(clock))

    def metadata(self):
        return dict(free=self.GPUTokenFree.copy(), prio=self.GPUTokenPriority.copy(),
                    idxbuf=self.GPUIndicesBuffer.copy(), to_host=self.GPUTokenToHost.copy(),
                    host_to_gpu=self.HostTokenToGPU.copy(), n_free=self.n_free, idx_count=self.idx_count)


# ---------------------------------------------------------------------------
# composite decode step (a0 append .. a5 EMA), in the order of the page's
# section 4 step list
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Reserve:
    """Direct-to-slot prefetch state: each recall sets aside `cap` slots; `slots` is
    the current reserve (the lowest-index free slots after the last recall)."""
    cap: int
    slots: np.ndarray = dataclasses.field(default_factory=lambda: np.zeros(0, np.int32))


def decode_step(pool: Pool, q, w, k_index, ctx_len, req_to_host, s_hat, k: int, clock: int,
                stage_stride: int, cap_div: int = 16, alpha: float = 0.5, new_kv=None,
                new_k_index=None, stats: Stats | None = None, staged=None, reserve: Reserve | None = None,
                assigned=None):
    """One layer's decode step on the oracle's own state (k_index, ctx_len, s_hat and
    pool are updated in place).  `staged` overrides the modelled prefetch set (the
    GPU's staged rows, for comparing stats); by default the candidate set truncated
    to the cap in token order is used.
    With `reserve` (direct-to-slot mode) prefetched rows go straight into the reserved
    slots: `assigned` = (slots, rows) as the GPU's tickets placed them, else the
    candidates in (request, token) order take the reserve in order; the per-request
    cap does not apply (the reserve bounds the prefetch).  Returns a dict of the
    step's outputs."""
    status = 0
    st = stats if stats is not None else Stats()
    if new_kv is not None:
        status |= pool.append(k_index, ctx_len, req_to_host, new_kv, new_k_index, clock, st)
    scores = indexer_score(q, w, k_index, ctx_len)
    cand, cap = prefetch_candidates(scores, s_hat, ctx_len, req_to_host, pool.HostTokenToGPU,
                                    stage_stride, cap_div)
    if reserve is not None:
        B = len(cand)
        if assigned is None:
            rows = np.concatenate([np.asarray(req_to_host[b][c], np.int32) for b, c in enumerate(cand)] +
                                  [np.zeros(0, np.int32)])
            n = min(rows.size, reserve.slots.size)
            if rows.size > n:
                status |= PREFETCH_CAP_HIT
            assigned = (reserve.slots[:n].copy(), rows[:n])
        slots_a, rows_a = (_arr(x, np.int32) for x in assigned)
        status |= pool.prefetch_direct(slots_a, rows_a, clock)
        staged = [rows_a] + [np.zeros(0, np.int32)] * (B - 1)   # the recall's count needs no request split
        sel, kth = select_topk(scores, ctx_len, k)
        out_slot, s2, reserve.slots = pool.prefetch_recall(sel, req_to_host, clock, staged=staged, stats=st,
                                                           reserve_cap=reserve.cap)
    else:
        if staged is None:
            staged = [np.asarray(req_to_host[b][c[:cap[b]]], np.int32) for b, c in enumerate(cand)]
        if any(len(c) > cp for c, cp in zip(cand, cap)):
            status |= PREFETCH_CAP_HIT
        sel, kth = select_topk(scores, ctx_len, k)
        out_slot, s2 = pool.prefetch_recall(sel, req_to_host, clock, staged=staged, stats=st)
    status |= s2
    s_hat[...] = ema_update(s_hat, kth, alpha)
    return dict(scores=scores, sel=sel, kth=kth, out_slot=out_slot, status=status, candidates=cand,
                cap=cap, staged=staged, stats=st)
