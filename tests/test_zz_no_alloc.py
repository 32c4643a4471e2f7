"""echo_prefetch_recall_noalloc: the recall for callers that cannot allocate device
memory (a runtime that has already handed all of HBM to weights and KV pools, or a
plugin that receives buffers but no allocator).  It runs on the library's own fixed
scratch instead of a caller workspace, so it must give exactly what the ordinary
recall gives on the same inputs -- and what the oracle's recall gives -- call after
call, without allocating anything.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from helpers import Case, dev

pytestmark = pytest.mark.gpu

MAX_SLOTS, MAX_ENTRIES = 262144, 32768   # the limits the header states for this call


def _selection(c: Case, seed: int):
    g = np.random.default_rng(seed)
    scores = g.standard_normal((c.B, c.n_q, c.L_max)).astype(np.float32)
    sel, _ = oracle.select_topk(scores, c.inp.ctx_len, c.k)
    return sel


@pytest.mark.parametrize("B,n_q,L,k,n_g,res", [
    (4, 1, 3000, 200, 1000, 1000),     # full pool: eviction on every call
    (3, 2, 2000, 300, 1500, 1400),     # two query tokens: repeated rows
])
def test_no_alloc_recall_equals_workspace_recall_twice(B, n_q, L, k, n_g, res):
    ref = Case(B, n_q, L, L, n_g, res, clock=100, seed=41, k=k)     # ordinary recall, caller workspace
    new = Case(B, n_q, L, L, n_g, res, clock=100, seed=41, k=k)     # same state, no workspace
    for call in range(2):
        sel = dev(_selection(ref, 500 + call))
        outs = []
        for c, fn in ((ref, "ws"), (new, "noalloc")):
            out = torch.full(tuple(sel.shape), -7, dtype=torch.int32, device="cuda")
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            stats = echo.Stats()
            if fn == "ws":
                echo.echo_prefetch_recall(c.pool, c.ws, sel, c.r2h_t, c.ctx, 100 + call, out, stats=stats,
                                          dev_status=st)
            else:
                echo.echo_prefetch_recall_noalloc(c.pool, sel, c.r2h_t, c.ctx, 100 + call, out, stats=stats,
                                                  dev_status=st)
            torch.cuda.synchronize()
            outs.append((out.cpu().numpy(), int(st.item()), stats.as_dict()))
        assert np.array_equal(outs[0][0], outs[1][0]), f"out_slot differs on call {call}"
        assert outs[0][1] == outs[1][1] and outs[0][2] == outs[1][2]
        m0, m1 = ref.gpu_meta(), new.gpu_meta()
        for key in m0:
            assert np.array_equal(m0[key], m1[key]), (call, key)
        assert torch.equal(ref.pool.gpu_kv, new.pool.gpu_kv)


def test_no_alloc_recall_matches_the_oracle_and_allocates_nothing():
    """Three calls in a row against the oracle's recall: out_slot, status, statistics,
    the five metadata arrays, the counters and every occupied slot's bytes.  After the
    first call (which resolves the scratch's address), the calls change neither the
    memory PyTorch holds nor the device's free memory."""
    c = Case(4, 1, 3000, 3000, 1000, 1000, clock=200, seed=43, k=200)
    for call in range(3):
        sel_np = _selection(c, 700 + call)
        sel = dev(sel_np)
        out = torch.full(tuple(sel.shape), -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        stats = echo.Stats()
        torch.cuda.synchronize()
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        echo.echo_prefetch_recall_noalloc(c.pool, sel, c.r2h_t, c.ctx, 200 + call, out, stats=stats,
                                          dev_status=st)
        torch.cuda.synchronize()
        alloc1, free1 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        if call > 0:
            assert alloc1 == alloc0, "the no-allocation recall changed PyTorch's allocations"
            assert free0 - free1 < (2 << 20), f"device free memory fell by {free0 - free1} bytes during the call"
        ostats = oracle.Stats()
        out_o, status_o = c.orc_pool.prefetch_recall(sel_np, c.r2h, 200 + call, stats=ostats)
        assert np.array_equal(out.cpu().numpy(), out_o), f"call {call}: out_slot differs from the oracle"
        assert int(st.item()) == status_o
        g, o = stats.as_dict(), ostats.as_dict()
        for key in ("selected", "unique_rows", "hits", "misses", "recalled", "unrecalled", "evicted"):
            assert g[key] == o[key], (call, key, g[key], o[key])
        c.assert_pool_equal(c.orc_pool, f"call {call}")


def test_no_alloc_recall_rejects_sizes_beyond_its_scratch():
    c = Case(1, 1, 40000, 40000, 1000, 100, clock=10, seed=42, k=40000)   # 40000 entries > 32768
    sel = torch.arange(40000, dtype=torch.int32, device="cuda").view(1, 1, 40000)
    out = torch.empty_like(sel)
    with pytest.raises(echo.EchoError, match="at most"):
        echo.echo_prefetch_recall_noalloc(c.pool, sel, c.r2h_t, c.ctx, 10, out)
    # a pool one slot larger than the scratch is laid out for
    host = torch.zeros((64, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    big = echo.Pool(MAX_SLOTS + 1, host)
    echo.echo_pool_init(big)
    r2h = torch.arange(64, dtype=torch.int32, device="cuda").view(1, 64)
    ctx = torch.tensor([64], dtype=torch.int32, device="cuda")
    sel = torch.arange(8, dtype=torch.int32, device="cuda").view(1, 1, 8)
    out = torch.full_like(sel, -7)
    with pytest.raises(echo.EchoError, match="at most"):
        echo.echo_prefetch_recall_noalloc(big, sel, r2h, ctx, 10, out)
    torch.cuda.synchronize()
    assert bool((out == -7).all()), "a rejected call wrote its output"


def test_no_alloc_recall_with_an_empty_batch():
    """B = 0: the call succeeds and the pool ends as the oracle's recall of an empty
    selection leaves it (the indices buffer lists this recall's allocations: none)."""
    c = Case(2, 1, 2000, 2000, 800, 700, clock=300, seed=44, k=100)
    sel = torch.empty((0, 1, 100), dtype=torch.int32, device="cuda")
    out = torch.empty_like(sel)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_prefetch_recall_noalloc(c.pool, sel, c.r2h_t[:0], c.ctx[:0], 300, out, dev_status=st)
    torch.cuda.synchronize()
    out_o, status_o = c.orc_pool.prefetch_recall(np.empty((0, 1, 100), np.int32), c.r2h[:0], 300)
    assert int(st.item()) == status_o == 0
    c.assert_pool_equal(c.orc_pool, "empty batch")
