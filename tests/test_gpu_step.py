"""The composite decode step (append -> indexer + fused prefetch -> top-k -> recall
-> EMA) against the oracle, step after step, eagerly and replayed from a CUDA graph.

Acceptance per stage: scores within 1e-3 relative; top-k bit-exact against the
oracle run on the GPU's own scores (and, against the oracle's scores, different
only at tokens within 1e-3 of the k-th score); recall metadata, out_slot and pool
bytes bit-exact against the oracle run on the GPU's selection; EMA bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import Case, SCORE_RTOL, assert_scores_close, dev

pytestmark = pytest.mark.gpu

RHO = 0.9


def near_tie_only(sel_gpu, sel_ref, ref_scores, kth_ref, ctx, n_q):
    """Tokens in one selection but not the other must lie within 1e-3 of the k-th score."""
    B = sel_gpu.shape[0]
    for b in range(B):
        for j in range(n_q):
            a = set(sel_gpu[b, j][sel_gpu[b, j] >= 0].tolist())
            r = set(sel_ref[b, j][sel_ref[b, j] >= 0].tolist())
            for p in a ^ r:
                assert abs(ref_scores[b, j, p] - kth_ref[b, j]) <= SCORE_RTOL * abs(kth_ref[b, j]) + 1e-6


class StepRunner:
    def __init__(self, c: Case, s_hat0, append: bool, prefetch=True):
        self.c = c
        self.out = echo.StepBuffers(c.B, c.n_q, c.L_max, c.k)
        self.s_hat = torch.full((c.B, c.n_q), s_hat0, dtype=torch.float32, device="cuda")
        self.clock = torch.tensor([c.clock], dtype=torch.int32, device="cuda")
        self.stats = echo.Stats()
        self.q_buf = c.q.clone()
        self.new_kv = torch.zeros((c.B, echo.KV_ELEMS), dtype=torch.int16, device="cuda") if append else None
        self.new_ki = torch.zeros((c.B, echo.D_INDEX), dtype=torch.uint8, device="cuda") if append else None
        self.args = echo.make_step_args(c.pool, c.ws, self.q_buf, c.w, c.k_index, c.ctx, c.r2h_t, c.k, self.out,
                                        stage=c.stage if prefetch else None, s_hat=self.s_hat,
                                        new_kv=self.new_kv, new_k_index=self.new_ki, clock_dev=self.clock,
                                        advance_clock=True, stats=self.stats)

    def set_inputs(self, q, kv=None, ki=None):
        self.q_buf.copy_(dev(q))
        if self.new_kv is not None:
            self.new_kv.copy_(dev(kv.view(np.int16)))
            self.new_ki.copy_(dev(ki))

    def run(self):
        echo.echo_decode_step(self.args)


def step_inputs(c: Case, step: int, q_float):
    qf, q = wl.next_query(q_float, RHO, c.seed, step)
    kv, ki = wl.new_tokens(c.B, c.seed, step)
    return qf, q, kv, ki


def check_step_against_oracle(c: Case, R: StepRunner, q, kv, ki, append, kI_o, ctx_o, s_hat_o, clock):
    torch.cuda.synchronize()
    O = c.orc_pool
    status_o = 0
    if append:
        status_o |= O.append(kI_o, ctx_o, c.r2h, kv, ki, clock)
    assert np.array_equal(c.ctx.cpu().numpy(), ctx_o)
    scores_g = R.out.scores.cpu().numpy()
    scores_o = oracle.indexer_score(q, c.inp.w, kI_o, ctx_o)
    valid = ~np.isnan(scores_o)
    assert_scores_close(scores_g[valid], scores_o[valid])
    sel_g, kth_g = R.out.sel.cpu().numpy(), R.out.kth.cpu().numpy()
    sel_og, kth_og = oracle.select_topk(scores_g, ctx_o, c.k)
    assert np.array_equal(sel_g, sel_og) and np.array_equal(kth_g, kth_og)
    sel_o, kth_o = oracle.select_topk(scores_o, ctx_o, c.k)
    near_tie_only(sel_g, sel_o, scores_o, kth_o, ctx_o, c.n_q)
    out_o, rs = O.prefetch_recall(sel_g, c.r2h, clock)
    status_o |= rs
    assert np.array_equal(R.out.out_slot.cpu().numpy(), out_o)
    c.assert_pool_equal(O, f"step clock {clock}")
    s_hat_o[...] = oracle.ema_update(s_hat_o, kth_g)
    assert np.array_equal(R.s_hat.cpu().numpy(), s_hat_o)
    st = int(R.out.dev_status.item()) & ~echo.DEV_PREFETCH_CAP_HIT
    assert st == status_o, (st, status_o)
    assert int(R.clock.item()) == clock + 1


@pytest.mark.parametrize("B,n_q,L,ctx0,k,n_g,res,append,seed", [
    (1, 1, 4096, 4096, 256, 1024, 512, False, 1),          # the tiny workload
    (4, 1, 3000, 2900, 256, 1200, 1200, True, 2),          # full pool, write-through append
    (3, 2, 2000, 1990, 200, 1500, 1400, True, 3),          # two query tokens
    (2, 1, 2501, 2480, 128, 900, 800, True, 4),            # rows of host rows not 16-byte aligned
])
def test_decode_steps_match_oracle(B, n_q, L, ctx0, k, n_g, res, append, seed):
    c = Case(B, n_q, L, ctx0, n_g, res, clock=1000, seed=seed, k=k)
    R = StepRunner(c, s_hat0=float("inf"), append=append)
    kI_o, ctx_o = c.inp.k_index.copy(), c.inp.ctx_len.copy()
    s_hat_o = np.full((B, n_q), np.inf, np.float32)
    qf = c.inp.q_float
    for step in range(4):
        qf, q, kv, ki = step_inputs(c, step, qf)
        R.set_inputs(q, kv, ki)
        R.out.dev_status.zero_()
        R.run()
        check_step_against_oracle(c, R, q, kv, ki, append, kI_o, ctx_o, s_hat_o, 1000 + step)


def test_decode_step_rows_beyond_the_claim_list_and_unstaged_host_rows():
    """Two top-k claim paths the workloads above do not reach: one CTA's slice holding
    more selected entries than its claim list (k = 4096 with every positive score in the
    first slice), and rows too long for the host rows of a slice to be staged in shared
    memory (L = 200000)."""
    for B, L, k, concentrate in ((2, 20000, 4096, True), (1, 200000, 2048, False)):
        c = Case(B, 1, L, L, 3 * B * k, 2 * B * k, clock=700, seed=41, k=k)
        if concentrate:
            ki = c.inp.k_index.copy()
            ki[:, L // 8:, :] = 0          # e4m3 code 0 is +0: these tokens score exactly 0
            c.inp.k_index[...] = ki
            c.k_index.copy_(dev(ki))
        R = StepRunner(c, s_hat0=float("inf"), append=False)
        kI_o, ctx_o = c.inp.k_index.copy(), c.inp.ctx_len.copy()
        s_hat_o = np.full((B, 1), np.inf, np.float32)
        qf = c.inp.q_float
        for step in range(2):
            qf, q, kv, ki2 = step_inputs(c, step, qf)
            R.set_inputs(q)
            R.out.dev_status.zero_()
            R.run()
            check_step_against_oracle(c, R, q, kv, ki2, False, kI_o, ctx_o, s_hat_o, 700 + step)


def test_prefetch_stages_exactly_the_candidates_tiny():
    """Tiny workload, threshold at the oracle's 90th-percentile score: the staged set is
    the candidate set (non-resident tokens scoring above the threshold, decided on the
    GPU's fp32 scores), and every staged row holds its host row's bytes."""
    c = Case(1, 1, 4096, 4096, 1024, 512, clock=1000, seed=11, k=256, cap_div=8)   # cap above the candidates
    ref = oracle.indexer_score(c.inp.q, c.inp.w, c.inp.k_index, c.inp.ctx_len)
    thr = np.float32(np.percentile(ref[0, 0], 90))
    s_hat = torch.full((1, 1), float(thr), device="cuda")
    scores = torch.empty((1, 1, 4096), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_indexer_score(c.q, c.w, c.k_index, c.ctx, scores, s_hat=s_hat, req_to_host=c.r2h_t, pool=c.pool,
                            stage=c.stage, dev_status=st)
    torch.cuda.synchronize()
    cand, cap = oracle.prefetch_candidates(scores.cpu().numpy(), s_hat.cpu().numpy(), c.inp.ctx_len, c.r2h,
                                           c.state.host_token_to_gpu, c.stage_stride, c.cap_div)
    n = int(c.stage.count[0])
    assert len(cand[0]) <= cap[0] and n == len(cand[0])
    rows = c.stage.host_row[0, :n].cpu().numpy()
    assert sorted(rows.tolist()) == sorted(c.r2h[0, cand[0]].tolist())
    assert np.array_equal(c.stage.rows[0, :n].cpu().numpy().view(np.uint16), c.host_np[rows])
    assert int(st.item()) == 0


def test_prefetch_cap_and_validity_under_minus_inf_threshold():
    """Threshold -inf: every non-resident token is a candidate; staging stops at the cap
    (ceil(L/16)), flags PREFETCH_CAP_HIT, and what it staged is valid."""
    B, L = 4, 20000
    c = Case(B, 1, L, L, 4000, 3000, clock=50, seed=12, k=512)
    s_hat = torch.full((B, 1), float("-inf"), device="cuda")
    scores = torch.empty((B, 1, L), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_indexer_score(c.q, c.w, c.k_index, c.ctx, scores, s_hat=s_hat, req_to_host=c.r2h_t, pool=c.pool,
                            stage=c.stage, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & echo.DEV_PREFETCH_CAP_HIT
    cap = min(c.stage_stride, -(-L // c.cap_div))
    for b in range(B):
        n = min(int(c.stage.count[b]), cap)
        rows = c.stage.host_row[b, :n].cpu().numpy()
        assert n == cap and len(set(rows.tolist())) == n
        assert np.all(c.state.host_token_to_gpu[rows] == echo.INF)
        assert np.all((rows >= b * L) & (rows < (b + 1) * L))
        assert np.array_equal(c.stage.rows[b, :n].cpu().numpy().view(np.uint16), c.host_np[rows])


def test_lossless_selection_and_pool_independent_of_the_prediction():
    """Section 6.1's lossless claim on the GPU: threshold -inf (prefetch up to the cap),
    +inf (no prefetch) and the EMA give identical selections, slots, metadata and bytes."""
    results = []
    # prediction -inf (stays -inf under the EMA: prefetch up to the cap every step),
    # no prefetch at all, and the EMA started from +inf
    for s0, prefetch in ((float("-inf"), True), (float("inf"), False), (float("inf"), True)):
        c = Case(2, 1, 6000, 6000, 3000, 3000, clock=500, seed=21, k=400)
        R = StepRunner(c, s_hat0=s0, append=True, prefetch=prefetch)
        qf = c.inp.q_float
        outs = []
        for step in range(4):
            qf, q, kv, ki = step_inputs(c, step, qf)
            R.set_inputs(q, kv, ki)
            R.run()
            torch.cuda.synchronize()
            outs.append((R.out.sel.cpu().numpy().copy(), R.out.out_slot.cpu().numpy().copy()))
        results.append((outs, c.gpu_meta(), c.pool.gpu_kv.cpu().numpy(), R.stats.as_dict()))
    for outs, meta, kv, stats in results[1:]:
        for (a, b), (x, y) in zip(results[0][0], outs):
            assert np.array_equal(a, x) and np.array_equal(b, y)
        for key in meta:
            assert np.array_equal(results[0][1][key], meta[key]), key
        assert np.array_equal(results[0][2], kv)
    assert results[0][3]["staged"] > 0 and results[1][3]["staged"] == 0 and results[2][3]["staged"] > 0


def test_graph_replay_equals_eager():
    """One captured graph replayed step after step (device clock) reproduces eager steps."""
    cases = [Case(2, 1, 3000, 2990, 1000, 1000, clock=300, seed=31, k=256) for _ in range(2)]
    runners = [StepRunner(c, s_hat0=float("inf"), append=True) for c in cases]
    qf = cases[0].inp.q_float
    seq = []
    for step in range(6):
        qf, q, kv, ki = step_inputs(cases[0], step, qf)
        seq.append((q, kv, ki))
    # step 0 eager on both (first calls set kernel attributes outside capture)
    for R in runners:
        R.set_inputs(*seq[0])
        R.run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            runners[1].run()
    torch.cuda.current_stream().wait_stream(s)
    for step in range(1, 6):
        runners[0].set_inputs(*seq[step])
        runners[0].run()
        runners[1].set_inputs(*seq[step])
        g.replay()
        torch.cuda.synchronize()
        a, b = runners
        for name in ("scores", "sel", "kth", "out_slot"):
            x, y = getattr(a.out, name).cpu().numpy(), getattr(b.out, name).cpu().numpy()
            assert np.array_equal(x, y, equal_nan=(name == "scores")), (step, name)
        ma, mb = cases[0].gpu_meta(), cases[1].gpu_meta()
        for key in ma:
            assert np.array_equal(ma[key], mb[key]), (step, key)
        assert torch.equal(cases[0].pool.gpu_kv, cases[1].pool.gpu_kv)
        assert torch.equal(a.s_hat, b.s_hat) and int(a.clock.item()) == int(b.clock.item()) == 301 + step


def test_stage_events_eager_and_captured():
    """Stage events (one record before each stage and one after the last) work on eager
    launches and inside a captured graph: the steps' outputs, the pool and the clock
    equal those of steps without events, and every stage's elapsed time is readable."""
    cases = [Case(2, 1, 3000, 2990, 1000, 1000, clock=300, seed=32, k=256) for _ in range(2)]
    plain = StepRunner(cases[0], s_hat0=float("inf"), append=False)
    timed = StepRunner(cases[1], s_hat0=float("inf"), append=False)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(echo.NUM_STAGES + 1)]
    for e in evs:
        e.record()
    c = cases[1]
    timed.args = echo.make_step_args(c.pool, c.ws, timed.q_buf, c.w, c.k_index, c.ctx, c.r2h_t, c.k, timed.out,
                                     stage=c.stage, s_hat=timed.s_hat, clock_dev=timed.clock, advance_clock=True,
                                     stats=timed.stats, events=evs)
    qf = cases[0].inp.q_float
    g = None
    for step in range(5):
        qf, q, _, _ = step_inputs(cases[0], step, qf)
        plain.set_inputs(q)
        plain.run()
        timed.set_inputs(q)
        if step < 3:       # eager: plain event records
            timed.run()
        else:              # captured once, then replayed: external event nodes
            if g is None:
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    with torch.cuda.graph(g, stream=s):
                        timed.run()
                torch.cuda.current_stream().wait_stream(s)
            g.replay()
        torch.cuda.synchronize()
        times = [evs[i].elapsed_time(evs[i + 1]) for i in range(echo.NUM_STAGES)]
        assert all(t >= 0.0 for t in times) and times[1] > 0.0, (step, times)
        for name in ("scores", "sel", "kth", "out_slot"):
            x, y = getattr(plain.out, name).cpu().numpy(), getattr(timed.out, name).cpu().numpy()
            assert np.array_equal(x, y, equal_nan=(name == "scores")), (step, name)
        ma, mb = cases[0].gpu_meta(), cases[1].gpu_meta()
        for key in ma:
            assert np.array_equal(ma[key], mb[key]), (step, key)
        assert torch.equal(plain.s_hat, timed.s_hat) and int(plain.clock.item()) == int(timed.clock.item())


def test_results_written_straight_into_pinned_host_memory():
    """out_slot and the status word may live in pinned host memory (zero-copy results):
    the same steps give the same slots, selections and pool as device-resident results."""
    runs = []
    for host_out in (False, True):
        c = Case(2, 1, 3000, 2990, 1000, 1000, clock=300, seed=41, k=256)
        R = StepRunner(c, s_hat0=float("inf"), append=True)
        if host_out:
            res = torch.zeros(2 * 256 + 1, dtype=torch.int32, pin_memory=True)
            R.out.out_slot = res[:2 * 256].view(2, 1, 256)
            R.out.dev_status = res[2 * 256:]
            R.args = echo.make_step_args(c.pool, c.ws, R.q_buf, c.w, c.k_index, c.ctx, c.r2h_t, c.k, R.out,
                                         stage=c.stage, s_hat=R.s_hat, new_kv=R.new_kv, new_k_index=R.new_ki,
                                         clock_dev=R.clock, advance_clock=True, stats=R.stats)
        qf = c.inp.q_float
        outs = []
        for step in range(4):
            qf, q, kv, ki = step_inputs(c, step, qf)
            R.set_inputs(q, kv, ki)
            R.run()
            torch.cuda.synchronize()
            outs.append((R.out.sel.cpu().numpy().copy(), R.out.out_slot.cpu().numpy().copy(),
                         int(R.out.dev_status.cpu().item())))
        runs.append((outs, c.gpu_meta(), c.pool.gpu_kv.cpu().numpy()))
    (a, ma, ka), (b, mb, kb) = runs
    for (s0, o0, st0), (s1, o1, st1) in zip(a, b):
        assert np.array_equal(s0, s1) and np.array_equal(o0, o1) and st0 == st1
        assert np.all(o1[s1 >= 0] >= 0)
    for key in ma:
        assert np.array_equal(ma[key], mb[key]), key
    assert np.array_equal(ka, kb)
