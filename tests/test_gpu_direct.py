"""Direct-to-slot prefetch on the GPU against the oracle.

The prefetch puts rows straight into GPU-pool slots that the previous recall set
aside.  Which candidate takes which reserved slot is decided by racing tickets, so
each test reads that assignment from the GPU (the first `staged` slots of the old
reserve, and the rows they now hold), checks that it is a valid one (distinct
candidate rows, as many as the reserve and the candidates allow, every byte equal to
the host row), hands it to the oracle, and then requires everything else to be
bit-exact: metadata, the next reserve, out_slot, statistics and pool bytes."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import Case, dev

pytestmark = pytest.mark.gpu

RHO = 0.9


def direct_case(B, n_q, L, ctx, n_g, res, clock, seed, k, R, while_scoring=False):
    c = Case(B, n_q, L, ctx, n_g, res, clock=clock, seed=seed, k=k)
    c.stage = echo.Stage(B, reserve=R, while_scoring=while_scoring)
    c.reserve = oracle.Reserve(R)
    return c


def check_reserve(c: Case):
    got = c.stage.reserved_slots()
    assert np.array_equal(got, c.reserve.slots), (got[:8], c.reserve.slots[:8])


def gpu_assignment(c: Case, old_reserve: np.ndarray, staged: int):
    slots = old_reserve[:staged].astype(np.int32)
    rows = c.pool.to_host[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy().astype(np.int32) \
        if staged else np.zeros(0, np.int32)
    return slots, rows


def check_assignment(c: Case, slots, rows, candidates, old_reserve, every=True):
    """every=False (prefetch while scoring): candidates still queued when scoring ended
    may be left out, so the placed rows are a subset of the candidates."""
    cand_rows = set()
    for b, toks in enumerate(candidates):
        cand_rows.update(int(c.r2h[b, p]) for p in toks)
    assert len(set(rows.tolist())) == rows.size, "a row placed twice"
    assert set(rows.tolist()) <= cand_rows, "a placed row was no candidate"
    want = min(len(old_reserve), len(cand_rows))
    assert rows.size == want if every else rows.size <= want, (rows.size, len(old_reserve), len(cand_rows))
    gkv = c.pool.gpu_kv.cpu().numpy().view(np.uint16)
    host = c.host_t.numpy().view(np.uint16)          # the live pool: appends write through
    assert np.array_equal(gkv[slots], host[rows])


def test_recall_builds_and_returns_the_reserve():
    """Recalls without any prefetch: the reserve is set aside, returned and set aside
    again, evicting for it; R = 0 returns it all."""
    c = direct_case(3, 1, 3000, 3000, 1500, 1450, clock=100, seed=51, k=200, R=300)
    g = np.random.default_rng(51)
    for step, R in enumerate((120, 120, 300, 0, 50)):
        c.stage.set_reserve_cap(R)
        c.reserve.cap = R
        scores = g.standard_normal((3, 1, 3000)).astype(np.float32)
        sel, _ = oracle.select_topk(scores, c.inp.ctx_len, 200)
        out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        stats = echo.Stats()
        echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, 100 + step, out, stage=c.stage,
                                  stats=stats, dev_status=st)
        ost = oracle.Stats()
        ref, rs, c.reserve.slots = c.orc_pool.prefetch_recall(sel, c.r2h, 100 + step, staged=[], stats=ost,
                                                              reserve_cap=R)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref)
        c.assert_pool_equal(c.orc_pool, f"recall {step}")
        check_reserve(c)
        assert int(st.item()) == rs
        assert stats.as_dict() == ost.as_dict()
        assert int(c.stage.reserve_ctl[0]) == 0


def test_indexer_fills_the_reserve_with_candidates_then_recall_matches_oracle():
    c = direct_case(2, 1, 4096, 4096, 2048, 1500, clock=300, seed=52, k=256, R=200)
    # the first reserve: a recall of an empty selection
    empty = np.full((2, 1, 256), -1, np.int32)
    out = torch.empty(empty.shape, dtype=torch.int32, device="cuda")
    echo.echo_prefetch_recall(c.pool, c.ws, dev(empty), c.r2h_t, c.ctx, 300, out, stage=c.stage)
    _, _, c.reserve.slots = c.orc_pool.prefetch_recall(empty, c.r2h, 300, reserve_cap=200)
    torch.cuda.synchronize()
    check_reserve(c)
    old = c.reserve.slots.copy()
    # the prefetch with the thresholds at the 95th and 99th percentile scores of the two
    # rows (about as many candidates as reserved slots)
    ref = oracle.indexer_score(c.inp.q, c.inp.w, c.inp.k_index, c.inp.ctx_len)
    thr = np.array([[np.percentile(ref[0, 0], 95)], [np.percentile(ref[1, 0], 99)]], np.float32)
    s_hat = dev(thr)
    scores = torch.empty((2, 1, 4096), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_indexer_score(c.q, c.w, c.k_index, c.ctx, scores, s_hat=s_hat, req_to_host=c.r2h_t, pool=c.pool,
                            stage=c.stage, dev_status=st)
    torch.cuda.synchronize()
    sc = scores.cpu().numpy()
    cand, _ = oracle.prefetch_candidates(sc, thr, c.inp.ctx_len, c.r2h, c.orc_pool.HostTokenToGPU, 4096, 1)
    n_cand = sum(len(x) for x in cand)
    taken = min(int(c.stage.reserve_ctl[0]), len(old))
    assert taken == min(n_cand, len(old))
    assert bool(int(st.item()) & echo.DEV_PREFETCH_CAP_HIT) == (n_cand > len(old))
    slots, rows = gpu_assignment(c, old, taken)
    check_assignment(c, slots, rows, cand, old)
    prio = c.pool.prio.cpu().numpy()
    assert np.all(prio[slots] == -3)        # filled this step, until the recall gives them its clock
    assert c.orc_pool.prefetch_direct(slots, rows, 301) == 0
    # the recall of the top-k selection
    sel, _ = oracle.select_topk(sc, c.inp.ctx_len, 256)
    out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = echo.Stats()
    echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, 301, out, stage=c.stage, stats=stats,
                              dev_status=st2)
    ost = oracle.Stats()
    ref_out, rs, c.reserve.slots = c.orc_pool.prefetch_recall(sel, c.r2h, 301, staged=[rows], stats=ost,
                                                              reserve_cap=200)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref_out)
    c.assert_pool_equal(c.orc_pool, "recall after the direct prefetch")
    check_reserve(c)
    assert int(st2.item()) == rs
    g, o = stats.as_dict(), ost.as_dict()
    assert g == o, (g, o)
    assert o["staged"] == taken and 0 < o["staged_used"] <= taken


class DirectRunner:
    def __init__(self, c: Case, append: bool, s_hat0=float("inf")):
        self.c = c
        self.out = echo.StepBuffers(c.B, c.n_q, c.L_max, c.k)
        self.s_hat = torch.full((c.B, c.n_q), s_hat0, dtype=torch.float32, device="cuda")
        self.clock = torch.tensor([c.clock], dtype=torch.int32, device="cuda")
        self.stats = echo.Stats()
        self.q_buf = c.q.clone()
        self.new_kv = torch.zeros((c.B, echo.KV_ELEMS), dtype=torch.int16, device="cuda") if append else None
        self.new_ki = torch.zeros((c.B, echo.D_INDEX), dtype=torch.uint8, device="cuda") if append else None
        self.args = echo.make_step_args(c.pool, c.ws, self.q_buf, c.w, c.k_index, c.ctx, c.r2h_t, c.k, self.out,
                                        stage=c.stage, s_hat=self.s_hat, new_kv=self.new_kv,
                                        new_k_index=self.new_ki, clock_dev=self.clock, advance_clock=True,
                                        stats=self.stats)

    def set_inputs(self, q, kv=None, ki=None):
        self.q_buf.copy_(dev(q))
        if self.new_kv is not None:
            self.new_kv.copy_(dev(kv.view(np.int16)))
            self.new_ki.copy_(dev(ki))

    def run(self):
        echo.echo_decode_step(self.args)

    def replay(self):
        """The step from one CUDA graph, captured at the first call."""
        if getattr(self, "graph", None) is None:
            self.graph = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                with torch.cuda.graph(self.graph, stream=s):
                    self.run()
            torch.cuda.current_stream().wait_stream(s)
        self.graph.replay()


@pytest.mark.parametrize("B,n_q,L,ctx0,k,n_g,res,R,append,seed,graph,ws", [
    (1, 1, 4096, 4096, 256, 1024, 512, 64, False, 61, False, False),     # the tiny workload
    (4, 1, 3000, 2900, 256, 1200, 1150, 300, True, 62, False, False),    # full pool: the reserve is evicted for
    (3, 2, 2000, 1990, 200, 1500, 1400, 100, True, 63, False, False),    # two query tokens
    (2, 1, 2501, 2480, 128, 900, 800, 900, True, 64, False, False),      # reserve larger than the pool can give
    (2, 1, 3000, 2990, 256, 1000, 1000, 250, True, 65, True, False),     # steps 1.. replayed from one graph
    (4, 1, 3000, 2900, 256, 1200, 1150, 300, True, 66, True, True),      # prefetch while scoring, graph
])
def test_direct_decode_steps_match_oracle(B, n_q, L, ctx0, k, n_g, res, R, append, seed, graph, ws):
    """The oracle follows the GPU step by step on the GPU's scores (the threshold test
    and the selection are decided in fp32; the scores themselves are compared with
    the oracle's in the staging-mode step tests).  Which reserved slot a prefetched
    row lands in is a race, so a graph replay is checked the same way, not against an
    eager run."""
    c = direct_case(B, n_q, L, ctx0, n_g, res, clock=1000, seed=seed, k=k, R=R, while_scoring=ws)
    run = DirectRunner(c, append)
    O = c.orc_pool
    kI_o, ctx_o = c.inp.k_index.copy(), c.inp.ctx_len.copy()
    s_hat_o = np.full((B, n_q), np.inf, np.float32)
    qf = c.inp.q_float
    used = 0
    for step in range(5):
        qf, q = wl.next_query(qf, RHO, seed, step)
        kv, ki = wl.new_tokens(B, seed, step)
        run.set_inputs(q, kv, ki)
        run.out.dev_status.zero_()
        old = c.reserve.slots.copy()
        staged0 = run.stats.as_dict()["staged"]
        if graph and step >= 1:
            run.replay()
        else:
            run.run()
        torch.cuda.synchronize()
        clock = 1000 + step
        status_o = 0
        if append:
            status_o |= O.append(kI_o, ctx_o, c.r2h, kv, ki, clock)
        assert np.array_equal(c.ctx.cpu().numpy(), ctx_o)
        scores_g = run.out.scores.cpu().numpy()
        cand, _ = oracle.prefetch_candidates(scores_g, s_hat_o, ctx_o, c.r2h, O.HostTokenToGPU, L, 1)
        slots, rows = gpu_assignment(c, old, run.stats.as_dict()["staged"] - staged0)
        check_assignment(c, slots, rows, cand, old, every=not ws)
        status_o |= O.prefetch_direct(slots, rows, clock)
        sel_g, kth_g = run.out.sel.cpu().numpy(), run.out.kth.cpu().numpy()
        sel_og, kth_og = oracle.select_topk(scores_g, ctx_o, k)
        assert np.array_equal(sel_g, sel_og) and np.array_equal(kth_g, kth_og)
        ost = oracle.Stats()
        out_o, rs, c.reserve.slots = O.prefetch_recall(sel_g, c.r2h, clock, staged=[rows], stats=ost,
                                                       reserve_cap=R)
        status_o |= rs
        assert np.array_equal(run.out.out_slot.cpu().numpy(), out_o)
        c.assert_pool_equal(O, f"direct step {step}")
        check_reserve(c)
        s_hat_o[...] = oracle.ema_update(s_hat_o, kth_g)
        assert np.array_equal(run.s_hat.cpu().numpy(), s_hat_o)
        st = int(run.out.dev_status.item()) & ~echo.DEV_PREFETCH_CAP_HIT
        assert st == status_o, (st, status_o)
        used += ost.as_dict()["staged_used"]
        assert int(run.clock.item()) == clock + 1
    g = run.stats.as_dict()
    assert g["staged_used"] == used
    assert g["staged"] > 0 and used > 0


def test_direct_lossless():
    """Selections are the same with the direct prefetch, the staging prefetch and no
    prefetch (each prefetch also while scoring only), and every selected token's slot
    holds its host row's bytes."""
    B, L, k, n_g, res = 2, 6000, 400, 3000, 2900
    runs = []
    for mode in ("direct", "staging", "none", "direct_while_scoring", "staging_while_scoring"):
        c = Case(B, 1, L, L - 10, n_g, res, clock=500, seed=71, k=k)
        if mode == "direct":
            c.stage = echo.Stage(B, reserve=500)
        if mode == "direct_while_scoring":
            c.stage = echo.Stage(B, reserve=500, while_scoring=True)
        if mode == "staging_while_scoring":
            c.stage = echo.Stage(B, c.stage_stride, c.cap_div, while_scoring=True)
        runner = DirectRunner(c, append=True, s_hat0=float("inf"))
        if mode == "none":
            runner.args = echo.make_step_args(c.pool, c.ws, runner.q_buf, c.w, c.k_index, c.ctx, c.r2h_t, k,
                                              runner.out, stage=None, s_hat=runner.s_hat, new_kv=runner.new_kv,
                                              new_k_index=runner.new_ki, clock_dev=runner.clock,
                                              advance_clock=True, stats=runner.stats)
        runs.append((mode, c, runner))
    qf = runs[0][1].inp.q_float
    for step in range(6):
        qf, q = wl.next_query(qf, RHO, 71, step)
        kv, ki = wl.new_tokens(B, 71, step)
        sels = []
        for mode, c, runner in runs:
            runner.set_inputs(q, kv, ki)
            runner.run()
            torch.cuda.synchronize()
            sel = runner.out.sel.cpu().numpy()
            slot = runner.out.out_slot.cpu().numpy()
            gkv = c.pool.gpu_kv.cpu().numpy().view(np.uint16)
            host = c.host_t.numpy().view(np.uint16)
            for b in range(B):
                ok = sel[b, 0] >= 0
                assert np.all(slot[b, 0][ok] >= 0)
                assert np.array_equal(gkv[slot[b, 0][ok]], host[c.r2h[b][sel[b, 0][ok]]])
            sels.append(sel)
        for (mode, _, _), sel in zip(runs[1:], sels[1:]):
            assert np.array_equal(sel, sels[0]), (step, mode)
    d = runs[0][2].stats.as_dict()
    s = runs[1][2].stats.as_dict()
    assert d["staged"] > 0 and s["staged"] > 0 and d["staged_used"] > 0
