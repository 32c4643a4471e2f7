"""The multi-step workload: 256 consecutive decode steps of 4 layers, batch 16, context
growing from 32K to 32K + 256 by one appended token per request per step (write-through
to the host pool and into a GPU slot), a 100K-slot GPU pool per layer that is full from
the start (the clock eviction runs every step), step-correlated queries (consecutive
top-k overlap 0.85).  All four layers' steps replay from one captured CUDA graph.

The oracle runs in lockstep on the GPU's selection: every step, every layer's out_slot
is bit-exact; every 32 steps the five metadata arrays and counters, the GPU-pool bytes
of every occupied slot, the EMA, the appended host rows, one request's scores (1e-3)
and two requests' top-k (bit-exact on the GPU's scores) are compared as well."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import assert_scores_close, dev, pinned_host_pool

pytestmark = pytest.mark.gpu

B, L0, STEPS, LAYERS, K, N_G, T0 = 16, 32768, 256, 4, 2048, 100_000, 1000
L_MAX = L0 + STEPS
N_H = B * L_MAX
RHO = 0.985418   # calibrated for overlap 0.85 at L = 32768 (tests/golden/rho_calibration.json)
CHECK_EVERY = 32


class Layer:
    def __init__(self, l: int, base_k: np.ndarray, base_host: np.ndarray, r2h_t):
        seed = 500 + l
        g = np.random.default_rng(seed)
        # this layer's keys: the base keys with the token positions permuted (cheap, distinct)
        perm = g.permutation(L_MAX)
        self.kI = np.ascontiguousarray(base_k[:, perm, :])
        self.ctx = np.full(B, L0, np.int32)
        inp = wl.indexer_inputs(B, 1, 1, 1, seed)   # q and w only (k^I above)
        self.w = inp.w
        self.qf = inp.q_float
        self.q0 = inp.q
        # host pool: the base pattern made distinct per layer
        host = base_host ^ np.uint16(0x1111 * (l + 1))
        self.host_t = pinned_host_pool(host)
        # GPU pool full at the start with random tokens of the first L0 positions
        idx = np.sort(g.choice(B * L0, size=N_G, replace=False))
        rows = (idx // L0) * L_MAX + idx % L0
        st = wl.resident_pool(N_G, N_H, rows, wl.random_clocks(N_G, T0, seed), seed)
        self.orc = oracle.Pool.from_state(st, host)
        self.pool = echo.Pool(N_G, self.host_t)
        self.pool.load_state(st)
        self.ws = echo.Workspace(N_G, B * K)
        self.stage = echo.Stage(B, (L_MAX + 15) // 16, 16)
        self.out = echo.StepBuffers(B, 1, L_MAX, K)
        self.stats = echo.Stats()
        self.s_hat = torch.full((B, 1), float("inf"), dtype=torch.float32, device="cuda")
        self.s_hat_o = np.full((B, 1), np.inf, np.float32)
        self.clock = torch.tensor([T0], dtype=torch.int32, device="cuda")
        self.q_buf = dev(self.q0)
        self.w_t = dev(self.w)
        self.k_t = dev(self.kI)
        self.ctx_t = dev(self.ctx)
        self.kv_buf = torch.zeros((B, echo.KV_ELEMS), dtype=torch.int16, device="cuda")
        self.ki_buf = torch.zeros((B, echo.D_INDEX), dtype=torch.uint8, device="cuda")
        self.args = echo.make_step_args(self.pool, self.ws, self.q_buf, self.w_t, self.k_t, self.ctx_t, r2h_t, K,
                                        self.out, stage=self.stage, s_hat=self.s_hat, new_kv=self.kv_buf,
                                        new_k_index=self.ki_buf, clock_dev=self.clock, advance_clock=True,
                                        stats=self.stats)
        self.seed = seed


def test_multi_step_four_layers_graph_replay_with_appends():
    base_k = wl.indexer_inputs(B, 1, L_MAX, L0, 499).k_index
    base_host = wl.host_kv_pool(N_H, 499, n_random=0)
    r2h = wl.req_to_host(B, L_MAX)
    r2h_t = dev(r2h)
    layers = [Layer(l, base_k, base_host, r2h_t) for l in range(LAYERS)]
    del base_k, base_host

    def set_inputs(t):
        for L in layers:
            if t > 0:
                L.qf, q = wl.next_query(L.qf, RHO, L.seed, t)
            else:
                q = L.q0
            kv, ki = wl.new_tokens(B, L.seed, t)
            L.q_buf.copy_(dev(q))
            L.kv_buf.copy_(dev(kv.view(np.int16)))
            L.ki_buf.copy_(dev(ki))
            L.cur = (q, kv, ki)

    def run_all():
        for L in layers:
            echo.echo_decode_step(L.args)

    # step 0 eagerly (first calls set kernel attributes), then one graph of all four layers
    set_inputs(0)
    run_all()
    torch.cuda.synchronize()
    check_step(layers, r2h, 0)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run_all()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in range(1, STEPS):
        set_inputs(t)
        g.replay()
        torch.cuda.synchronize()
        check_step(layers, r2h, t)
    for L in layers:
        assert int(L.clock.item()) == T0 + STEPS
        assert np.array_equal(L.ctx_t.cpu().numpy(), np.full(B, L0 + STEPS, np.int32))
        st = L.stats.as_dict()
        assert st["steps"] == STEPS and st["appended"] == STEPS * B and st["unrecalled"] == 0
        assert st["evicted"] >= st["recalled"] > 0
        # the library's own invariant check finds every pool consistent after the run
        report = torch.zeros(len(echo.VAL_FIELDS), dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_pool_validate(L.pool, report, status)
        torch.cuda.synchronize()
        rep = dict(zip(echo.VAL_FIELDS, report.cpu().tolist()))
        assert int(status.item()) == 0, rep
        assert rep["occupied"] == N_G - int(L.pool.counters[0]) == rep["resident"], rep


def check_step(layers, r2h, t):
    clock = T0 + t
    full = (t % CHECK_EVERY == CHECK_EVERY - 1) or t == 0
    for li, L in enumerate(layers):
        q, kv, ki = L.cur
        status = L.orc.append(L.kI, L.ctx, r2h, kv, ki, clock)
        sel = L.out.sel.cpu().numpy()
        out_o, rs = L.orc.prefetch_recall(sel, r2h, clock)
        status |= rs
        assert np.array_equal(L.out.out_slot.cpu().numpy(), out_o), f"layer {li} step {t}: out_slot differs"
        st = int(L.out.dev_status.item()) & ~echo.DEV_PREFETCH_CAP_HIT
        assert st == status, (li, t, st, status)
        kth = L.out.kth.cpu().numpy()
        L.s_hat_o[...] = oracle.ema_update(L.s_hat_o, kth)
        if not full:
            continue
        # metadata, counters and bytes against the lockstep oracle
        m, o = L.pool.metadata(), L.orc.metadata()
        for key in ("free", "prio", "idxbuf", "to_host", "host_to_gpu", "n_free", "idx_count"):
            assert np.array_equal(m[key], o[key]), f"layer {li} step {t}: {key} differs"
        occ = np.nonzero(o["free"] == 0)[0]
        gkv = L.pool.gpu_kv.cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv[occ], L.orc.gpu_kv[occ]), f"layer {li} step {t}: GPU-pool bytes differ"
        assert np.array_equal(gkv[occ], L.orc.host_kv[o["to_host"][occ]])
        assert np.array_equal(L.s_hat.cpu().numpy(), L.s_hat_o)
        # the appended rows reached the pinned host pool and the indexer cache
        p = L0 + t
        rows = r2h[:, p]
        assert np.array_equal(L.host_t.numpy().view(np.uint16)[rows], kv)
        assert np.array_equal(L.k_t[:, p, :].cpu().numpy(), ki)
        # every selected row is resident, at the slot out_slot names
        slot = L.out.out_slot.cpu().numpy()
        valid = sel >= 0
        assert np.all(slot[valid] >= 0)
        hrow = np.take_along_axis(np.broadcast_to(r2h[:, None, :], (B, 1, L_MAX)), np.where(valid, sel, 0), axis=2)
        assert np.array_equal(m["to_host"][slot[valid]], hrow[valid])
        # one layer per check: one request's scores against the oracle, two requests' top-k
        if li == (t // CHECK_EVERY) % len(layers):
            b = (t // CHECK_EVERY) % B
            scores_g = L.out.scores.cpu().numpy()
            ctx = L.ctx
            ref = oracle.indexer_score(q[b:b + 1], L.w[b:b + 1], L.kI[b:b + 1], ctx[b:b + 1])
            n = int(ctx[b])
            assert_scores_close(scores_g[b, 0, :n], ref[0, 0, :n], f"layer {li} step {t} scores")
            for bb in (b, (b + 7) % B):
                sel_o, kth_o = oracle.select_topk(scores_g[bb:bb + 1], ctx[bb:bb + 1], K)
                assert np.array_equal(sel[bb:bb + 1], sel_o) and np.array_equal(kth[bb:bb + 1], kth_o)
