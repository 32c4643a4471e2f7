"""GB300 (sm_103a) ECHO decode step: thin ctypes binding over libecho_gb300.

Every function here marshals arguments (torch tensors -> raw pointers, the
current CUDA stream) and calls the C ABI of include/echo.h with the same name;
all work runs in the library's CUDA kernels.  There is no CPU or PyTorch
fallback: importing the binding without the built library raises.

Buffers are plain torch tensors: device tensors for the GPU side, a pinned
(page-locked, mapped) CPU tensor for the host KV pool.  `Pool`, `Workspace`,
`Stage` and `Stats` are small holders that allocate those tensors and build the
C structs.
"""
from __future__ import annotations

import ctypes
import os
import platform

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, f"libecho_gb300_{platform.machine()}.so")

ECHO_OK, ECHO_EINVAL, ECHO_ECUDA, ECHO_ENOTSUP = 0, 1, 2, 3
DEV_POOL_EXHAUSTED, DEV_BAD_INDEX, DEV_WAIT_TIMEOUT, DEV_PREFETCH_CAP_HIT, DEV_INVARIANT = 1, 2, 4, 8, 16
VAL_FIELDS = ("slot_state", "slot_map", "row_map", "counter", "reserve", "free", "occupied", "reserved",
              "resident", "reserve_balance")
INF = 0x7FFFFFFF
H_INDEX, D_INDEX, KV_ELEMS, KV_BYTES = 64, 128, 576, 1152
STAGE_APPEND, STAGE_INDEXER, STAGE_TOPK, STAGE_RECALL, STAGE_EMA, NUM_STAGES = range(6)
STAT_FIELDS = ("steps", "selected", "unique_rows", "hits", "misses", "recalled", "unrecalled",
               "evicted", "staged", "staged_used", "appended")

_P = ctypes.c_void_p
_I32 = ctypes.c_int32


class EchoError(RuntimeError):
    pass


class c_pool(ctypes.Structure):
    _fields_ = [("n_g", _I32), ("n_h", _I32), ("gpu_token_free", _P), ("gpu_token_priority", _P),
                ("gpu_indices_buffer", _P), ("gpu_token_to_host", _P), ("host_token_to_gpu", _P),
                ("gpu_kv", _P), ("host_kv", _P), ("counters", _P), ("row_elems", _I32)]


class c_workspace(ctypes.Structure):
    _fields_ = [("base", _P), ("bytes", ctypes.c_size_t), ("n_g", _I32), ("max_rows", _I32)]


class c_stage(ctypes.Structure):
    _fields_ = [("rows", _P), ("host_row", _P), ("count", _P), ("stride", _I32), ("cap_div", _I32),
                ("reserve", _P), ("reserve_ctl", _P), ("reserve_cap", _I32), ("flags", _I32)]


class c_indexer_args(ctypes.Structure):
    _fields_ = [("q", _P), ("w", _P), ("k_index", _P), ("ctx_len", _P), ("B", _I32), ("n_q", _I32),
                ("L_max", _I32), ("scores", _P), ("s_hat", _P), ("req_to_host", _P),
                ("pool", ctypes.POINTER(c_pool)), ("stage", ctypes.POINTER(c_stage)), ("dev_status", _P)]


class c_prefill_args(ctypes.Structure):
    _fields_ = [("q", _P), ("w", _P), ("k_index", _P), ("ctx_len", _P), ("B", _I32), ("C", _I32),
                ("L_max", _I32), ("scores", _P), ("s_shift", _P), ("k", _I32), ("thr_bin", _P), ("subset_n", _P),
                ("req_to_host", _P), ("pool", ctypes.POINTER(c_pool)), ("stage", ctypes.POINTER(c_stage)),
                ("dev_status", _P)]


class c_mla_args(ctypes.Structure):
    _fields_ = [("q", _P), ("gpu_kv", _P), ("n_g", _I32), ("out_slot", _P), ("B", _I32), ("n_q", _I32),
                ("k", _I32), ("scale", ctypes.c_float), ("out", _P), ("lse", _P), ("workspace", _P),
                ("workspace_bytes", ctypes.c_size_t), ("dev_status", _P)]


class c_step_args(ctypes.Structure):
    _fields_ = [("pool", ctypes.POINTER(c_pool)), ("ws", ctypes.POINTER(c_workspace)),
                ("stage", ctypes.POINTER(c_stage)), ("q", _P), ("w", _P), ("k_index", _P), ("ctx_len", _P),
                ("req_to_host", _P), ("B", _I32), ("n_q", _I32), ("L_max", _I32), ("k", _I32),
                ("scores", _P), ("sel", _P), ("kth", _P), ("out_slot", _P), ("s_hat", _P),
                ("alpha", ctypes.c_float), ("new_kv", _P), ("new_k_index", _P), ("clock", _I32),
                ("clock_dev", _P), ("advance_clock", _I32), ("stats", _P), ("dev_status", _P),
                ("stage_events", ctypes.POINTER(_P))]


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise EchoError(f"libecho_gb300 is not built ({path}); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    S = ctypes.c_int
    sig = {
        "echo_indexer_score": ([ctypes.POINTER(c_indexer_args), _P], S),
        "echo_select_topk": ([_P, _P, _I32, _I32, _I32, _I32, _P, _P, _P], S),
        "echo_workspace_bytes": ([_I32, _I32, ctypes.POINTER(ctypes.c_size_t)], S),
        "echo_selftest_wait_timeout": ([_I32, _P, _P], S),
        "echo_workspace_init": ([ctypes.POINTER(c_workspace), _P], S),
        "echo_pool_init": ([ctypes.POINTER(c_pool), _P], S),
        "echo_pool_alloc": ([ctypes.POINTER(c_pool), ctypes.POINTER(c_workspace), _P, _P, _I32, _I32, _P, _P, _P, _P], S),
        "echo_pool_evict": ([ctypes.POINTER(c_pool), ctypes.POINTER(c_workspace), _P, _I32, _P, _P, _P], S),
        "echo_prefetch_recall": ([ctypes.POINTER(c_pool), ctypes.POINTER(c_workspace), _P, _P, _P, _I32, _I32, _I32,
                                  _I32, ctypes.POINTER(c_stage), _I32, _P, _P, _P, _P, _P], S),
        "echo_append": ([ctypes.POINTER(c_pool), ctypes.POINTER(c_workspace), _P, _P, _P, _I32, _I32, _P, _P, _I32,
                         _P, _P, _P, _P], S),
        "echo_prefetch_recall_noalloc": ([ctypes.POINTER(c_pool), _P, _P, _P, _I32, _I32, _I32, _I32,
                                          ctypes.POINTER(c_stage), _I32, _P, _P, _P, _P, _P], S),
        "echo_ema_update": ([_P, _P, _I32, ctypes.c_float, _P], S),
        "echo_ema_update_strided": ([_P, _P, _I32, _I32, ctypes.c_float, _P], S),
        "echo_prefill_indexer_score": ([ctypes.POINTER(c_prefill_args), _P], S),
        "echo_mla_workspace_bytes": ([_I32, _I32, _I32, ctypes.POINTER(ctypes.c_size_t)], S),
        "echo_sparse_mla_decode": ([ctypes.POINTER(c_mla_args), _P], S),
        "echo_decode_step": ([ctypes.POINTER(c_step_args), _P], S),
        "echo_decode_step_host": ([ctypes.POINTER(c_step_args), _P, _P, _P, _I32], S),
        "echo_step_graph_create": ([ctypes.POINTER(c_step_args), ctypes.POINTER(_P)], S),
        "echo_step_graph_launch": ([_P, _P, _P, _P, _I32], S),
        "echo_step_graph_destroy": ([_P], S),
        "echo_pool_validate": ([ctypes.POINTER(c_pool), ctypes.POINTER(c_stage), _P, _P, _P], S),
        "echo_pool_validate_host": ([ctypes.POINTER(c_pool), _P, _I32, _P], S),
        "echo_last_error_string": ([], ctypes.c_char_p),
        "echo_version": ([], _I32),
        "echo_metadata_bytes": ([ctypes.c_int64, ctypes.c_int64], ctypes.c_int64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != ECHO_OK:
        msg = load_library().echo_last_error_string().decode()
        raise EchoError(f"{what} failed (code {rc}): {msg}")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise EchoError("tensors passed to libecho_gb300 must be contiguous")
    return t.data_ptr()


def _dev(t: torch.Tensor | None, name: str):
    if t is not None and not t.is_cuda:
        raise EchoError(f"{name} must be a CUDA tensor")
    return _ptr(t)


def _current_stream_handle():
    return torch.cuda.current_stream().cuda_stream


try:  # the raw handle of the current stream without building a Stream object
    _raw_stream, _cur_device = torch._C._cuda_getCurrentRawStream, torch._C._cuda_getDevice

    def _current_stream_handle():  # noqa: F811
        return _raw_stream(_cur_device())
except AttributeError:
    pass


def _stream(stream):
    if stream is None:
        return _current_stream_handle()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ---------------------------------------------------------------------------
# holders
# ---------------------------------------------------------------------------

class Pool:
    """One layer's GPU pool plus a view of the (per-model) pinned host pool.  A row is
    host_kv's last dimension: 576 (MLA's latent row of one token) or, for the
    block-level / GQA variant, any multiple of 8 up to 65536 bf16 (a block of tokens
    of one KV head)."""

    def __init__(self, n_g: int, host_kv: torch.Tensor, device="cuda"):
        if host_kv.device.type != "cpu" or not host_kv.is_pinned():
            raise EchoError("host_kv must be a pinned CPU tensor")
        R = int(host_kv.shape[-1]) if host_kv.dim() == 2 else -1
        if host_kv.dtype not in (torch.int16, torch.uint16, torch.bfloat16) or R <= 0 or R % 8 or R > 65536:
            raise EchoError("host_kv must be [n_h][R] 16-bit with R a multiple of 8 up to 65536")
        self.n_g = int(n_g)
        self.n_h = int(host_kv.shape[0])
        self.row_elems = R
        self.host_kv = host_kv
        self.free = torch.empty(n_g, dtype=torch.uint8, device=device)
        self.prio = torch.empty(n_g, dtype=torch.int32, device=device)
        self.idxbuf = torch.empty(n_g, dtype=torch.int32, device=device)
        self.to_host = torch.empty(n_g, dtype=torch.int32, device=device)
        self.host_to_gpu = torch.empty(self.n_h, dtype=torch.int32, device=device)
        self.gpu_kv = torch.zeros((n_g, R), dtype=torch.int16, device=device)
        self.counters = torch.zeros(4, dtype=torch.int32, device=device)
        self.c = c_pool(self.n_g, self.n_h, _ptr(self.free), _ptr(self.prio), _ptr(self.idxbuf),
                        _ptr(self.to_host), _ptr(self.host_to_gpu), _ptr(self.gpu_kv), _ptr(host_kv),
                        _ptr(self.counters), R)

    def load_state(self, st, gpu_kv=None):
        """Install a workload.PoolState (metadata arrays + counters); gpu_kv defaults
        to the host rows of the occupied slots."""
        import numpy as np
        self.free.copy_(torch.from_numpy(st.gpu_token_free))
        self.prio.copy_(torch.from_numpy(st.gpu_token_priority))
        self.idxbuf.copy_(torch.from_numpy(st.gpu_indices_buffer))
        self.to_host.copy_(torch.from_numpy(st.gpu_token_to_host))
        self.host_to_gpu.copy_(torch.from_numpy(st.host_token_to_gpu))
        self.counters.copy_(torch.tensor([st.n_free, st.idx_count, 0, 0], dtype=torch.int32))
        if gpu_kv is None:
            occ = np.nonzero(st.gpu_token_free == 0)[0]
            kv = torch.zeros((self.n_g, self.row_elems), dtype=torch.int16)
            if occ.size:
                hk = self.host_kv.view(torch.int16)
                kv[torch.from_numpy(occ)] = hk[torch.from_numpy(st.gpu_token_to_host[occ].astype(np.int64))]
            self.gpu_kv.copy_(kv)
        else:
            self.gpu_kv.copy_(gpu_kv)

    def metadata(self):
        return dict(free=self.free.cpu().numpy(), prio=self.prio.cpu().numpy(), idxbuf=self.idxbuf.cpu().numpy(),
                    to_host=self.to_host.cpu().numpy(), host_to_gpu=self.host_to_gpu.cpu().numpy(),
                    n_free=int(self.counters[0]), idx_count=int(self.counters[1]))


class Workspace:
    def __init__(self, n_g: int, max_rows: int, device="cuda", stream=None):
        n = ctypes.c_size_t()
        _check(load_library().echo_workspace_bytes(n_g, max_rows, ctypes.byref(n)), "echo_workspace_bytes")
        self.buf = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
        base = (self.buf.data_ptr() + 255) & ~255
        self.c = c_workspace(base, n.value, n_g, max_rows)
        _check(load_library().echo_workspace_init(ctypes.byref(self.c), _stream(stream)), "echo_workspace_init")


class Stage:
    """Where the prefetch puts rows: a staging area of `stride` rows per request, or,
    with reserve=R, straight into R GPU-pool slots each recall sets aside (direct to
    slot; the staging buffers are not allocated then).  while_scoring: the decode
    indexer drops candidates still queued when a CTA's scoring ends."""

    def __init__(self, B: int, stride: int = 1, cap_div: int = 16, device="cuda", reserve: int | None = None,
                 while_scoring: bool = False):
        self.direct = reserve is not None
        self.stride, self.cap_div = int(stride), int(cap_div)
        self.count = torch.zeros(B, dtype=torch.int32, device=device)
        if self.direct:
            self.rows = self.host_row = None
            self.reserve_cap = int(reserve)
            self.reserve = torch.full((max(self.reserve_cap, 1),), -1, dtype=torch.int32, device=device)
            self.reserve_ctl = torch.zeros(2, dtype=torch.int32, device=device)
            self.c = c_stage(None, None, _ptr(self.count), self.stride, self.cap_div, _ptr(self.reserve),
                             _ptr(self.reserve_ctl), self.reserve_cap, int(bool(while_scoring)))
        else:
            self.rows = torch.zeros((B, stride, KV_ELEMS), dtype=torch.int16, device=device)
            self.host_row = torch.full((B, stride), -1, dtype=torch.int32, device=device)
            self.reserve = self.reserve_ctl = None
            self.reserve_cap = 0
            self.c = c_stage(_ptr(self.rows), _ptr(self.host_row), _ptr(self.count), self.stride, self.cap_div,
                             None, None, 0, int(bool(while_scoring)))

    def set_reserve_cap(self, R: int):
        """Slots each recall sets aside from now on (at most the capacity allocated)."""
        if not self.direct or not 0 <= R <= self.reserve.numel():
            raise EchoError(f"reserve_cap {R} outside [0, {self.reserve.numel()}] or stage not direct")
        self.reserve_cap = int(R)
        self.c.reserve_cap = int(R)

    def reserved_slots(self):
        """The current reserve (direct to slot), as a numpy array."""
        n = int(self.reserve_ctl[1])
        return self.reserve[:n].cpu().numpy()


class Stats:
    def __init__(self, device="cuda"):
        self.t = torch.zeros(len(STAT_FIELDS), dtype=torch.int64, device=device)

    def as_dict(self):
        v = self.t.cpu().tolist()
        return dict(zip(STAT_FIELDS, v))


# ---------------------------------------------------------------------------
# C-ABI calls
# ---------------------------------------------------------------------------

def echo_indexer_score(q, w, k_index, ctx_len, scores, s_hat=None, req_to_host=None, pool: Pool | None = None,
                       stage: Stage | None = None, dev_status=None, stream=None):
    B, n_q = q.shape[0], q.shape[1]
    a = c_indexer_args(_dev(q, "q"), _dev(w, "w"), _dev(k_index, "k_index"), _dev(ctx_len, "ctx_len"), B, n_q,
                       k_index.shape[1], _dev(scores, "scores"), _dev(s_hat, "s_hat"),
                       _dev(req_to_host, "req_to_host"),
                       ctypes.pointer(pool.c) if pool is not None else None,
                       ctypes.pointer(stage.c) if stage is not None else None, _dev(dev_status, "dev_status"))
    _check(load_library().echo_indexer_score(ctypes.byref(a), _stream(stream)), "echo_indexer_score")


def echo_prefill_indexer_score(q, w, k_index, ctx_len, scores, s_shift=None, k: int = 0, thr_bin=None,
                               subset_n=None, req_to_host=None, pool: Pool | None = None,
                               stage: Stage | None = None, dev_status=None, stream=None):
    """q [B][C][64][128] e4m3: the chunk's C queries per request (see include/echo.h)."""
    B, C = q.shape[0], q.shape[1]
    a = c_prefill_args(_dev(q, "q"), _dev(w, "w"), _dev(k_index, "k_index"), _dev(ctx_len, "ctx_len"), B, C,
                       k_index.shape[1], _dev(scores, "scores"), _dev(s_shift, "s_shift"), int(k),
                       _dev(thr_bin, "thr_bin"), _dev(subset_n, "subset_n"), _dev(req_to_host, "req_to_host"),
                       ctypes.pointer(pool.c) if pool is not None else None,
                       ctypes.pointer(stage.c) if stage is not None else None, _dev(dev_status, "dev_status"))
    _check(load_library().echo_prefill_indexer_score(ctypes.byref(a), _stream(stream)),
           "echo_prefill_indexer_score")


def echo_select_topk(scores, ctx_len, k: int, sel, kth, stream=None):
    B, n_q, L_max = scores.shape
    _check(load_library().echo_select_topk(_dev(scores, "scores"), _dev(ctx_len, "ctx_len"), B, n_q, L_max, k,
                                           _dev(sel, "sel"), _dev(kth, "kth"), _stream(stream)), "echo_select_topk")


def echo_pool_init(pool: Pool, stream=None):
    _check(load_library().echo_pool_init(ctypes.byref(pool.c), _stream(stream)), "echo_pool_init")


def echo_pool_alloc(pool: Pool, ws: Workspace, host_idx, n_dev, clock: int, out_slots, dev_status=None,
                    clock_dev=None, stream=None):
    _check(load_library().echo_pool_alloc(ctypes.byref(pool.c), ctypes.byref(ws.c), _dev(host_idx, "host_idx"),
                                          _dev(n_dev, "n_dev"), int(host_idx.numel()), int(clock),
                                          _dev(clock_dev, "clock_dev"), _dev(out_slots, "out_slots"),
                                          _dev(dev_status, "dev_status"), _stream(stream)), "echo_pool_alloc")


def echo_pool_evict(pool: Pool, ws: Workspace, n_needed_dev, clock: int, dev_status=None, clock_dev=None,
                    stream=None):
    _check(load_library().echo_pool_evict(ctypes.byref(pool.c), ctypes.byref(ws.c), _dev(n_needed_dev, "n_needed"),
                                          int(clock), _dev(clock_dev, "clock_dev"), _dev(dev_status, "dev_status"),
                                          _stream(stream)), "echo_pool_evict")


def echo_prefetch_recall(pool: Pool, ws: Workspace, sel, req_to_host, ctx_len, clock: int, out_slot,
                         stage: Stage | None = None, stats: Stats | None = None, dev_status=None, clock_dev=None,
                         stream=None):
    B, n_q, k = sel.shape
    _check(load_library().echo_prefetch_recall(
        ctypes.byref(pool.c), ctypes.byref(ws.c), _dev(sel, "sel"), _dev(req_to_host, "req_to_host"),
        _dev(ctx_len, "ctx_len"), B, n_q, k, req_to_host.shape[1],
        ctypes.pointer(stage.c) if stage is not None else None, int(clock), _dev(clock_dev, "clock_dev"),
        _dev(out_slot, "out_slot"), _dev(stats.t, "stats") if stats is not None else None,
        _dev(dev_status, "dev_status"), _stream(stream)), "echo_prefetch_recall")


def echo_prefetch_recall_noalloc(pool: Pool, sel, req_to_host, ctx_len, clock: int, out_slot,
                                 stage: Stage | None = None, stats: Stats | None = None, dev_status=None,
                                 clock_dev=None, stream=None):
    """Guaranteed recall without a caller workspace (the library's own fixed scratch)."""
    B, n_q, k = sel.shape
    _check(load_library().echo_prefetch_recall_noalloc(
        ctypes.byref(pool.c), _dev(sel, "sel"), _dev(req_to_host, "req_to_host"), _dev(ctx_len, "ctx_len"), B, n_q,
        k, req_to_host.shape[1], ctypes.pointer(stage.c) if stage is not None else None, int(clock),
        _dev(clock_dev, "clock_dev"), _dev(out_slot, "out_slot"), _dev(stats.t, "stats") if stats is not None else None,
        _dev(dev_status, "dev_status"), _stream(stream)), "echo_prefetch_recall_noalloc")


def echo_selftest_wait_timeout(which: int, dev_status, stream=None):
    """A wait nothing satisfies gives up after a second and flags WAIT_TIMEOUT."""
    _check(load_library().echo_selftest_wait_timeout(int(which), _dev(dev_status, "dev_status"), _stream(stream)),
           "echo_selftest_wait_timeout")


def echo_append(pool: Pool, ws: Workspace, k_index, ctx_len, req_to_host, new_kv, new_k_index, clock: int,
                stats: Stats | None = None, dev_status=None, clock_dev=None, stream=None):
    B, L_max = k_index.shape[0], k_index.shape[1]
    _check(load_library().echo_append(
        ctypes.byref(pool.c), ctypes.byref(ws.c), _dev(k_index, "k_index"), _dev(ctx_len, "ctx_len"),
        _dev(req_to_host, "req_to_host"), B, L_max, _dev(new_kv, "new_kv"), _dev(new_k_index, "new_k_index"),
        int(clock), _dev(clock_dev, "clock_dev"), _dev(stats.t, "stats") if stats is not None else None,
        _dev(dev_status, "dev_status"), _stream(stream)), "echo_append")


def echo_ema_update(s_hat, kth, alpha: float = 0.5, stream=None):
    _check(load_library().echo_ema_update(_dev(s_hat, "s_hat"), _dev(kth, "kth"), int(s_hat.numel()),
                                          float(alpha), _stream(stream)), "echo_ema_update")


class MlaWorkspace:
    """Scratch of echo_sparse_mla_decode for B requests, n_q queries, k selected rows."""

    def __init__(self, B: int, n_q: int, k: int, device="cuda"):
        n = ctypes.c_size_t()
        _check(load_library().echo_mla_workspace_bytes(B, n_q, k, ctypes.byref(n)), "echo_mla_workspace_bytes")
        self.buf = torch.empty(n.value + 256, dtype=torch.uint8, device=device)
        self.base = (self.buf.data_ptr() + 255) & ~255
        self.bytes = n.value


def echo_sparse_mla_decode(q, gpu_kv, out_slot, scale: float, out, lse, ws: MlaWorkspace, dev_status=None,
                           stream=None):
    """q [B][n_q][128][576] bf16 (int16 bits), gpu_kv [n_g][576] (the pool's rows),
    out_slot [B][n_q][k]; out [B][n_q][128][512] fp32, lse [B][n_q][128] fp32."""
    B, n_q, k = out_slot.shape
    a = c_mla_args(_dev(q, "q"), _dev(gpu_kv, "gpu_kv"), int(gpu_kv.shape[0]), _dev(out_slot, "out_slot"), B, n_q,
                   k, float(scale), _dev(out, "out"), _dev(lse, "lse"), ws.base, ws.bytes,
                   _dev(dev_status, "dev_status"))
    _check(load_library().echo_sparse_mla_decode(ctypes.byref(a), _stream(stream)), "echo_sparse_mla_decode")


def echo_ema_update_strided(s_hat, kth, kth_stride: int, alpha: float = 0.5, stream=None):
    """s_hat[i] from kth[i * kth_stride] (kth a flat device tensor view)."""
    _check(load_library().echo_ema_update_strided(_dev(s_hat, "s_hat"), _dev(kth, "kth"), int(s_hat.numel()),
                                                  int(kth_stride), float(alpha), _stream(stream)),
           "echo_ema_update_strided")


class StepBuffers:
    """Device outputs of one decode step for B requests, n_q queries, k."""

    def __init__(self, B: int, n_q: int, L_max: int, k: int, device="cuda"):
        # entries past each row's context are never written: NaN marks them
        self.scores = torch.full((B, n_q, L_max), float("nan"), dtype=torch.float32, device=device)
        self.sel = torch.empty((B, n_q, k), dtype=torch.int32, device=device)
        self.kth = torch.empty((B, n_q), dtype=torch.float32, device=device)
        self.out_slot = torch.empty((B, n_q, k), dtype=torch.int32, device=device)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=device)


def make_step_args(pool: Pool, ws: Workspace, q, w, k_index, ctx_len, req_to_host, k: int, out: StepBuffers,
                   stage: Stage | None = None, s_hat=None, alpha: float = 0.5, new_kv=None, new_k_index=None,
                   clock: int = 0, clock_dev=None, advance_clock: bool = False, stats: Stats | None = None,
                   events=None) -> c_step_args:
    """Build the C struct once (e.g. before graph capture); keep the returned object
    alive while it is in use."""
    B, n_q = q.shape[0], q.shape[1]
    a = c_step_args()
    a.pool = ctypes.pointer(pool.c)
    a.ws = ctypes.pointer(ws.c)
    a.stage = ctypes.pointer(stage.c) if stage is not None else None
    a.q, a.w, a.k_index = _dev(q, "q"), _dev(w, "w"), _dev(k_index, "k_index")
    a.ctx_len, a.req_to_host = _dev(ctx_len, "ctx_len"), _dev(req_to_host, "req_to_host")
    a.B, a.n_q, a.L_max, a.k = B, n_q, k_index.shape[1], int(k)
    a.scores, a.sel, a.kth, a.out_slot = _ptr(out.scores), _ptr(out.sel), _ptr(out.kth), _ptr(out.out_slot)
    a.s_hat = _dev(s_hat, "s_hat")
    a.alpha = float(alpha)
    a.new_kv, a.new_k_index = _dev(new_kv, "new_kv"), _dev(new_k_index, "new_k_index")
    a.clock = int(clock)
    a.clock_dev = _dev(clock_dev, "clock_dev")
    a.advance_clock = 1 if advance_clock else 0
    a.stats = _dev(stats.t, "stats") if stats is not None else None
    a.dev_status = _ptr(out.dev_status)
    if events is not None:
        arr = (_P * (NUM_STAGES + 1))(*[e.cuda_event for e in events])
        a._events_keepalive = arr
        a.stage_events = arr
    # keep the referenced holders alive with the struct
    a._keep = (pool, ws, stage, q, w, k_index, ctx_len, req_to_host, out, s_hat, new_kv, new_k_index, clock_dev,
               stats)
    return a


def echo_pool_validate(pool: Pool, report, dev_status, stage: Stage | None = None, stream=None):
    """Metadata invariants on the device: report [len(VAL_FIELDS)] int32 (device) gets the
    counts, DEV_INVARIANT is OR-ed into dev_status when one is broken."""
    _check(load_library().echo_pool_validate(ctypes.byref(pool.c), ctypes.pointer(stage.c) if stage is not None
                                             else None, _dev(report, "report"), _dev(dev_status, "dev_status"),
                                             _stream(stream)), "echo_pool_validate")


def echo_pool_validate_host(free, prio, to_host, host_to_gpu, n_free: int, reserve=None):
    """The same invariants over host copies (numpy arrays: free uint8 [n_g], prio /
    to_host int32 [n_g], host_to_gpu int32 [n_h]).  Returns (violation found, counts)."""
    import numpy as np
    arrs = [np.ascontiguousarray(free, np.uint8), np.ascontiguousarray(prio, np.int32),
            np.ascontiguousarray(to_host, np.int32), np.ascontiguousarray(host_to_gpu, np.int32)]
    counters = np.array([n_free, 0, 0, 0], np.int32)
    idx = np.full(arrs[0].size, -1, np.int32)
    res = None if reserve is None else np.ascontiguousarray(reserve, np.int32)
    report = np.zeros(len(VAL_FIELDS), np.int32)
    ptr = lambda a: a.ctypes.data if a is not None and a.size else None
    c = c_pool(arrs[0].size, arrs[3].size, ptr(arrs[0]), ptr(arrs[1]), ptr(idx), ptr(arrs[2]), ptr(arrs[3]),
               None, None, ptr(counters), 0)
    rc = load_library().echo_pool_validate_host(ctypes.byref(c), ptr(res), 0 if res is None else res.size,
                                                ptr(report))
    if rc < 0:
        _check(-rc, "echo_pool_validate_host")
    return rc == DEV_INVARIANT, dict(zip(VAL_FIELDS, report.tolist()))


def echo_decode_step(args: c_step_args, stream=None):
    _check((_lib or load_library()).echo_decode_step(ctypes.byref(args), _stream(stream)), "echo_decode_step")


def _host_inputs(q_host, w_host):
    for t, name in ((q_host, "q_host"), (w_host, "w_host")):
        if t.is_cuda or not t.is_contiguous():
            raise EchoError(f"{name} must be a contiguous host tensor")
    return q_host.data_ptr(), w_host.data_ptr()


def echo_decode_step_host(args: c_step_args, q_host, w_host, stream=None, wait: bool = True):
    """One decode step whose q and w come from host tensors (pinned for an asynchronous
    copy) laid out as the step's device q and w; wait: return after the step is done."""
    qp, wp = _host_inputs(q_host, w_host)
    _check((_lib or load_library()).echo_decode_step_host(ctypes.byref(args), qp, wp, _stream(stream),
                                                          1 if wait else 0), "echo_decode_step_host")


class StepGraph:
    """A decode step captured into a CUDA graph by the library (echo_step_graph_*).
    The step's arguments (and every buffer they name) are kept alive with it."""

    def __init__(self, args: c_step_args):
        h = _P()
        _check(load_library().echo_step_graph_create(ctypes.byref(args), ctypes.byref(h)), "echo_step_graph_create")
        self._h, self._args = h, args

    def launch(self, q_host=None, w_host=None, stream=None, wait: bool = True):
        qp, wp = _host_inputs(q_host, w_host) if q_host is not None else (None, None)
        _check(_lib.echo_step_graph_launch(self._h, qp, wp, _stream(stream), 1 if wait else 0),
               "echo_step_graph_launch")

    def close(self):
        if self._h:
            _check(_lib.echo_step_graph_destroy(self._h), "echo_step_graph_destroy")
            self._h = _P()

    def __del__(self):
        try:
            if self._h and _lib is not None:
                _lib.echo_step_graph_destroy(self._h)
        except Exception:
            pass


def version() -> int:
    return int(load_library().echo_version())
