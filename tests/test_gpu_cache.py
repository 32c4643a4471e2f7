"""Cache manager and guaranteed recall on the GPU against the oracle: metadata,
out_slot, statistics and GPU-pool bytes bit-exact on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import Case, dev, pinned_host_pool

pytestmark = pytest.mark.gpu


def test_pool_init_and_alloc_match_oracle():
    n_g, n_h = 1000, 5000
    host = wl.host_kv_pool(n_h, 1)
    ht = pinned_host_pool(host)
    P = echo.Pool(n_g, ht)
    echo.echo_pool_init(P)
    ws = echo.Workspace(n_g, 512)
    O = oracle.Pool.empty(n_g, n_h, host.copy())
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = np.random.default_rng(1)
    for it, n in enumerate((300, 0, 512, 400)):
        rows = g.integers(0, n_h, size=512).astype(np.int32)
        rows[5] = rows[3]          # a repeat
        rows[7] = -4               # out of range
        out = torch.empty(512, dtype=torch.int32, device="cuda")
        echo.echo_pool_alloc(P, ws, dev(rows), dev(np.array([n], np.int32)), 10 + it, out, dev_status=st)
        ref, rstatus = O.alloc(rows[:n], 10 + it)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy()[:n], ref)
        m, o = P.metadata(), O.metadata()
        for key in o:
            assert np.array_equal(m[key], o[key]), (it, key)
        assert (int(st.item()) & rstatus) == rstatus


def test_evict_matches_oracle_and_moves_no_bytes():
    c = Case(B=2, n_q=1, L_max=3000, ctx=3000, n_g=2000, n_resident=1900, clock=50, seed=3, k=64)
    O = c.orc_pool
    kv0 = c.pool.gpu_kv.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for n, clock in ((0, 50), (37, 50), (600, 51), (5000, 52)):
        echo.echo_pool_evict(c.pool, c.ws, dev(np.array([n], np.int32)), clock, dev_status=st)
        ne, rs = O.evict(n, clock)
        torch.cuda.synchronize()
        c.assert_pool_equal(O, f"evict {n}")
    assert int(st.item()) & echo.DEV_POOL_EXHAUSTED
    assert torch.equal(c.pool.gpu_kv, kv0)


def recall_and_compare(c: Case, sel: np.ndarray, clock: int, stage_rows=None):
    out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
    stats = echo.Stats()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, clock, out,
                              stage=c.stage if stage_rows is not None else None, stats=stats, dev_status=st)
    ost = oracle.Stats()
    ref, rstatus = c.orc_pool.prefetch_recall(sel, c.r2h, clock, staged=stage_rows, stats=ost)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref)
    c.assert_pool_equal(c.orc_pool, "recall")
    assert int(st.item()) == rstatus
    g, o = stats.as_dict(), ost.as_dict()
    assert g == o, (g, o)
    return out


@pytest.mark.parametrize("B,n_q,L,k,n_g,res,seed", [
    (1, 1, 4096, 256, 1024, 512, 1),       # the tiny workload: pool half full
    (4, 1, 3000, 200, 1000, 1000, 2),      # full pool: eviction every step
    (3, 2, 2000, 300, 1500, 1400, 3),      # two query tokens: de-duplicated union
    (2, 1, 5000, 700, 900, 880, 4),        # misses exceed the pool: exhaustion
    (4, 1, 8192, 1024, 40000, 2000, 5),    # mostly free, over 128 slots per CTA: the misses take
                                           # the free slots of a few CTAs, copies spread over the grid
])
def test_recall_matches_oracle(B, n_q, L, k, n_g, res, seed):
    c = Case(B, n_q, L, L, n_g, res, clock=100, seed=seed, k=k)
    g = np.random.default_rng(seed)
    for step in range(3):
        scores = g.standard_normal((B, n_q, L)).astype(np.float32)
        sel, _ = oracle.select_topk(scores, c.inp.ctx_len, k)
        recall_and_compare(c, sel, clock=100 + step)


def test_recall_uses_staged_rows_bytes_exact():
    """Rows the prefetch staged are copied from the staging area; bytes still equal the host rows."""
    c = Case(2, 1, 2000, 2000, 600, 500, clock=20, seed=6, k=150)
    sel, _ = oracle.select_topk(np.random.default_rng(6).standard_normal((2, 1, 2000)).astype(np.float32),
                                c.inp.ctx_len, 150)
    staged = []
    for b in range(2):
        rows = [int(c.r2h[b, p]) for p in sel[b, 0][:60] if c.state.host_token_to_gpu[c.r2h[b, p]] == echo.INF]
        rows += [int(c.r2h[b, 1999 - i]) for i in range(10)]      # staged but not selected
        rows = [r for r in dict.fromkeys(rows) if c.state.host_token_to_gpu[r] == echo.INF][:c.stage_stride]
        staged.append(rows)
        c.stage.host_row[b, :len(rows)] = torch.tensor(rows, dtype=torch.int32)
        c.stage.rows[b, :len(rows)] = torch.from_numpy(c.host_np[rows].view(np.int16)).cuda()
        c.stage.count[b] = len(rows)
    recall_and_compare(c, sel, 20, stage_rows=staged)
    assert int(c.stage.count.sum()) == 0   # reset for the next step


def test_append_matches_oracle():
    B, L = 3, 500
    c = Case(B, 1, L, [200, 499, 10], 300, 300, clock=9, seed=7, k=32)
    kI = c.inp.k_index.copy()
    ctx = c.inp.ctx_len.copy()
    for step in range(3):
        kv, kn = wl.new_tokens(B, 7, step)
        stats = echo.Stats()
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_append(c.pool, c.ws, c.k_index, c.ctx, c.r2h_t, dev(kv.view(np.int16)), dev(kn), 9 + step,
                         stats=stats, dev_status=st)
        ost = oracle.Stats()
        rs = c.orc_pool.append(kI, ctx, c.r2h, kv, kn, 9 + step, ost)
        torch.cuda.synchronize()
        assert int(st.item()) == rs
        assert np.array_equal(c.ctx.cpu().numpy(), ctx)
        assert np.array_equal(c.k_index.cpu().numpy(), kI)
        assert np.array_equal(c.host_t.numpy().view(np.uint16), c.orc_pool.host_kv)
        c.assert_pool_equal(c.orc_pool, f"append {step}")
        assert stats.as_dict()["appended"] == ost.as_dict()["appended"]
        assert stats.as_dict()["evicted"] == ost.as_dict()["evicted"]


def test_append_of_a_resident_row_matches_oracle():
    """A caller state in which a new token's host row is already resident: both sides
    write the row through, flag BAD_INDEX, and take or free no slot for it."""
    B, L = 3, 400
    c = Case(B, 1, L, [100, 200, 300], 200, 199, clock=9, seed=8, k=32)
    future = np.array([c.r2h[0, 100]], np.int32)            # request 0's next token
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    echo.echo_pool_alloc(c.pool, c.ws, dev(future), dev(np.array([1], np.int32)), 9, out)
    slots, rs0 = c.orc_pool.alloc(future, 9)
    torch.cuda.synchronize()
    assert rs0 == 0 and int(out.item()) == int(slots[0])
    kI, ctx = c.inp.k_index.copy(), c.inp.ctx_len.copy()
    kv, kn = wl.new_tokens(B, 8, 0)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = echo.Stats()
    echo.echo_append(c.pool, c.ws, c.k_index, c.ctx, c.r2h_t, dev(kv.view(np.int16)), dev(kn), 10, stats=stats,
                     dev_status=st)
    ost = oracle.Stats()
    rs = c.orc_pool.append(kI, ctx, c.r2h, kv, kn, 10, ost)
    torch.cuda.synchronize()
    assert rs & oracle.BAD_INDEX and int(st.item()) == rs
    assert np.array_equal(c.ctx.cpu().numpy(), ctx) and np.array_equal(c.k_index.cpu().numpy(), kI)
    assert np.array_equal(c.host_t.numpy().view(np.uint16), c.orc_pool.host_kv)
    c.assert_pool_equal(c.orc_pool, "append with a resident row")
    assert stats.as_dict()["appended"] == ost.as_dict()["appended"] == 2
    assert stats.as_dict()["evicted"] == ost.as_dict()["evicted"] == 2


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_gives_up_and_the_context_stays_usable(which):
    """A wait nothing satisfies (an mbarrier with no arrivals; a grid barrier one CTA
    never reaches) gives up after about a second with WAIT_TIMEOUT; work launched
    afterwards runs normally."""
    import time
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    echo.echo_selftest_wait_timeout(which, st)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) & echo.DEV_WAIT_TIMEOUT
    assert 0.5 < dt < 30.0
    c = Case(1, 1, 512, 512, 64, 32, clock=5, seed=9, k=16)
    scores = torch.empty((1, 1, 512), dtype=torch.float32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_indexer_score(c.q, c.w, c.k_index, c.ctx, scores, dev_status=st2)
    torch.cuda.synchronize()
    ref = oracle.indexer_score(c.inp.q, c.inp.w, c.inp.k_index, c.inp.ctx_len)
    assert int(st2.item()) == 0
    assert np.allclose(scores.cpu().numpy(), ref, rtol=1e-3, atol=1e-6)


def _barrier_words(ws: echo.Workspace):
    """The grid barrier's arrival count and generation inside a recall workspace: the
    scratch layout puts 256-byte-aligned int32 arrays in this order: slot claims [n_g],
    nine per-entry arrays [max_rows], histograms [4][4096], per-CTA counts [1024][4],
    then the global words (arrival count at index 2, generation at index 5)."""
    a = lambda n: (n * 4 + 255) // 256 * 256
    off = (ws.c.base - ws.buf.data_ptr()) + a(ws.c.n_g) + 9 * a(ws.c.max_rows) + a(4 * 4096) + a(1024 * 4)
    glob = ws.buf[off:off + 64].view(torch.int32)
    return glob


def test_recalls_across_the_barrier_generation_wrap_match_oracle():
    """The cache manager's grid barrier counts arrivals back to zero at every barrier
    and numbers its generations modulo 2^32: with the generation word set just below
    the wrap, consecutive recalls still match the oracle and leave the arrival count
    at rest."""
    c = Case(4, 1, 3000, 3000, 1000, 1000, clock=400, seed=46, k=200)
    glob = _barrier_words(c.ws)
    torch.cuda.synchronize()
    assert int(glob[2]) == 0 and int(glob[5]) == 0       # a fresh workspace
    glob[5] = -3                                          # 0xFFFFFFFD: wraps within the next calls
    g = np.random.default_rng(46)
    for call in range(4):
        scores = g.standard_normal((c.B, 1, c.L_max)).astype(np.float32)
        sel_np, _ = oracle.select_topk(scores, c.inp.ctx_len, c.k)
        out = torch.full(sel_np.shape, -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_prefetch_recall(c.pool, c.ws, dev(sel_np), c.r2h_t, c.ctx, 400 + call, out, dev_status=st)
        torch.cuda.synchronize()
        out_o, status_o = c.orc_pool.prefetch_recall(sel_np, c.r2h, 400 + call)
        assert np.array_equal(out.cpu().numpy(), out_o), f"call {call}"
        assert int(st.item()) == status_o
        c.assert_pool_equal(c.orc_pool, f"call {call}")
        assert int(glob[2]) == 0, "the arrival count did not return to rest"
    assert 0 <= int(glob[5]) < 100, "the generation did not wrap"
