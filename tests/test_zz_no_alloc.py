"""echo_prefetch_recall_noalloc: the recall for callers that cannot allocate device
memory (a runtime that has already handed all of HBM to weights and KV pools, or a
plugin that receives buffers but no allocator).  It runs on the library's own fixed
scratch instead of a caller workspace, so it must give exactly what the ordinary
recall gives on the same inputs, call after call.

Kept in a file of its own that pytest collects last."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from helpers import Case, dev

pytestmark = pytest.mark.gpu


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


def test_no_alloc_recall_rejects_sizes_beyond_its_scratch():
    c = Case(1, 1, 40000, 40000, 1000, 100, clock=10, seed=42, k=40000)   # 40000 entries > 32768
    sel = torch.arange(40000, dtype=torch.int32, device="cuda").view(1, 1, 40000)
    out = torch.empty_like(sel)
    with pytest.raises(echo.EchoError, match="at most"):
        echo.echo_prefetch_recall_noalloc(c.pool, sel, c.r2h_t, c.ctx, 10, out)
