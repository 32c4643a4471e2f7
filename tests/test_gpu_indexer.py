"""Indexer score (tcgen05 FP8 kernel) against the oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import assert_scores_close, dev

pytestmark = pytest.mark.gpu


def run_indexer(inp, L_max, fill=float("nan")):
    B, n_q = inp.q.shape[:2]
    scores = torch.full((B, n_q, L_max), fill, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_indexer_score(dev(inp.q), dev(inp.w), dev(inp.k_index), dev(inp.ctx_len), scores, dev_status=st)
    torch.cuda.synchronize()
    return scores.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("B,n_q,L_max,ctx", [
    (1, 1, 4096, [4096]),                 # the tiny workload
    (3, 1, 1000, [1000, 1, 257]),         # ragged: partial tiles, a 1-token request
    (2, 2, 777, [777, 130]),              # two query tokens (MTP), causal by query
    (4, 1, 640, [0, 640, 0, 129]),        # empty requests
    (5, 2, 2048, [2048, 2047, 128, 129, 1]),
])
def test_indexer_matches_oracle(B, n_q, L_max, ctx):
    inp = wl.indexer_inputs(B, n_q, L_max, ctx, seed=B * 100 + L_max)
    got, status = run_indexer(inp, L_max)
    ref = oracle.indexer_score(inp.q, inp.w, inp.k_index, inp.ctx_len)
    assert status == 0
    valid = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~valid)   # entries past each query's length untouched
    assert_scores_close(got[valid], ref[valid])


def test_indexer_special_values():
    """All-zero q gives exact zeros; negated q gives ReLU of the negated dots."""
    inp = wl.indexer_inputs(2, 1, 300, [300, 300], seed=5)
    inp.q[0] = 0
    inp.q[1] ^= np.uint8(0x80)
    got, _ = run_indexer(inp, 300)
    assert np.all(got[0] == 0.0)
    ref = oracle.indexer_score(inp.q, inp.w, inp.k_index, inp.ctx_len)
    assert_scores_close(got[1], ref[1])


def test_indexer_deepseek_shape_sampled():
    """B=8, L=64K (the DeepSeek-V3.2 decode shape): every tile's first and last token
    and a random sample, each recomputed by the oracle one by one."""
    B, L = 8, 65536
    inp = wl.indexer_inputs(B, 1, L, L, seed=2)
    got, status = run_indexer(inp, L)
    assert status == 0 and not np.isnan(got).any()
    g = np.random.default_rng(0)
    pts = [(b, p) for b in range(B) for p in (0, 127, 128, L - 129, L - 128, L - 1)]
    pts += [(int(b), int(p)) for b, p in zip(g.integers(0, B, 600), g.integers(0, L, 600))]
    ref = np.array([oracle.indexer_score_one(inp.q, inp.w, inp.k_index, b, 0, p) for b, p in pts])
    assert_scores_close(np.array([got[b, 0, p] for b, p in pts]), ref)


def test_indexer_mtp_large_sampled():
    """n_q = 2 at B=4, L=100000 (HBM-pressure shape, fewer requests)."""
    B, L = 4, 100000
    ctx = [100000, 99999, 50000, 77777]
    inp = wl.indexer_inputs(B, 2, L, ctx, seed=3)
    got, status = run_indexer(inp, L)
    assert status == 0
    g = np.random.default_rng(1)
    pts = []
    for b in range(B):
        for j in range(2):
            v = ctx[b] - (1 - j)
            pts += [(b, j, 0), (b, j, v - 1)] + [(b, j, int(p)) for p in g.integers(0, v, 60)]
            if v < L:
                assert np.isnan(got[b, j, v:]).all()
    ref = np.array([oracle.indexer_score_one(inp.q, inp.w, inp.k_index, b, j, p) for b, j, p in pts])
    assert_scores_close(np.array([got[b, j, p] for b, j, p in pts]), ref)
