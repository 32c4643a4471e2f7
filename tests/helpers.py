"""Shared setup for the GPU parity tests: seeded inputs from the workload module,
the same bytes handed to the CUDA library (through the binding) and to the oracle."""
import numpy as np
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl

SCORE_RTOL = 1e-3   # fp32 tensor-core accumulation vs the fp64 oracle (relative)


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def pinned_host_pool(host_np: np.ndarray) -> torch.Tensor:
    t = torch.empty(host_np.shape, dtype=torch.int16, pin_memory=True)
    t.numpy()[...] = host_np.view(np.int16)
    return t


def stamp_host_rows(hv: np.ndarray):
    """Fill a [n][R] uint16 host pool so that every 16-byte vector of every row is
    distinct: elements 0-1 hold the row index, element 2 the vector's index in the
    row, the rest a bf16 1.0.  A copy that moves only part of a row, takes a vector
    from the wrong row, or shifts vectors within a row leaves a visible difference."""
    n, R = hv.shape
    v = hv.reshape(n, R // 8, 8)
    ids = np.arange(n, dtype=np.uint32)
    v[:, :, 0] = (ids & np.uint32(0xFFFF)).astype(np.uint16)[:, None]
    v[:, :, 1] = (ids >> np.uint32(16)).astype(np.uint16)[:, None]
    v[:, :, 2] = np.arange(R // 8, dtype=np.uint16)[None, :]
    v[:, :, 3:] = 0x3F80


def assert_recall_stats_equal(gpu: dict, orc: dict, msg=""):
    """The recall's counters that do not depend on the prefetch's timing."""
    for key in ("steps", "selected", "unique_rows", "hits", "misses", "recalled", "unrecalled", "evicted"):
        assert gpu[key] == orc[key], f"{msg} stats {key}: gpu {gpu[key]} oracle {orc[key]}"


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, what="scores"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = SCORE_RTOL * np.maximum(np.abs(ref), 1e-6)
    bad = np.abs(gpu - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} outside 1e-3 relative, e.g. gpu={gpu[bad][:4]} ref={ref[bad][:4]}"


class Case:
    """One layer: indexer inputs, pools (GPU + oracle copies), request->host map."""

    def __init__(self, B, n_q, L_max, ctx, n_g, n_resident, clock, seed, k, n_h=None, stage_stride=None,
                 cap_div=16, scatter=True):
        self.B, self.n_q, self.L_max, self.k, self.clock, self.seed = B, n_q, L_max, k, clock, seed
        self.inp = wl.indexer_inputs(B, n_q, L_max, ctx, seed)
        self.n_h = n_h or B * L_max
        self.host_np = wl.host_kv_pool(self.n_h, seed, n_random=min(self.n_h, B * L_max))
        self.r2h = wl.req_to_host(B, L_max)
        # resident rows are rows of tokens that exist: position p < ctx of their request
        ctx_b = np.broadcast_to(np.asarray(ctx, np.int64), (B,))
        exist = np.concatenate([b * L_max + np.arange(int(ctx_b[b]), dtype=np.int64) for b in range(B)])
        exist = exist[exist < self.n_h]
        rows = np.sort(exist[wl.random_resident_rows(exist.size, min(n_resident, exist.size), seed)])
        self.state = wl.resident_pool(n_g, self.n_h, rows, wl.random_clocks(n_resident, clock, seed), seed,
                                      scatter=scatter)
        self.host_t = pinned_host_pool(self.host_np)
        self.pool = echo.Pool(n_g, self.host_t)
        self.pool.load_state(self.state)
        self.ws = echo.Workspace(n_g, max(B * n_q * k, B))
        self.stage_stride = stage_stride or max(1, (L_max + cap_div - 1) // cap_div)
        self.stage = echo.Stage(B, self.stage_stride, cap_div)
        self.cap_div = cap_div
        self.q = dev(self.inp.q)
        self.w = dev(self.inp.w)
        self.k_index = dev(self.inp.k_index)
        self.ctx = dev(self.inp.ctx_len)
        self.r2h_t = dev(self.r2h)
        self.orc_pool = oracle.Pool.from_state(self.state, self.host_np.copy())

    def gpu_meta(self):
        return self.pool.metadata()

    def assert_pool_equal(self, orc: "oracle.Pool", msg=""):
        m = self.gpu_meta()
        o = orc.metadata()
        for key in ("free", "prio", "idxbuf", "to_host", "host_to_gpu", "n_free", "idx_count"):
            a, b = m[key], o[key]
            assert np.array_equal(a, b), f"{msg} metadata {key} differs at {np.nonzero(np.asarray(a) != np.asarray(b))[0][:8] if np.ndim(a) else (a, b)}"
        occ = np.nonzero(o["free"] == 0)[0]
        gkv = self.pool.gpu_kv.cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv[occ], orc.gpu_kv[occ]), f"{msg} GPU pool bytes differ"
