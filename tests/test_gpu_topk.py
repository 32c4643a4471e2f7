"""Exact top-k (cluster radix select): bit-exact against the oracle on the same scores."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from helpers import dev

pytestmark = pytest.mark.gpu


def gpu_topk(scores: np.ndarray, ctx, k):
    B, n_q, L = scores.shape
    sel = torch.full((B, n_q, k), -7, dtype=torch.int32, device="cuda")
    kth = torch.zeros((B, n_q), dtype=torch.float32, device="cuda")
    echo.echo_select_topk(dev(scores.astype(np.float32)), dev(np.asarray(ctx, np.int32)), k, sel, kth)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), kth.cpu().numpy()


def check(scores, ctx, k):
    sel, kth = gpu_topk(scores, ctx, k)
    rsel, rkth = oracle.select_topk(scores, ctx, k)
    assert np.array_equal(sel, rsel), f"sel differs in {np.argwhere((sel != rsel).any(axis=2))[:4]}"
    assert np.array_equal(kth.view(np.uint32), rkth.view(np.uint32)) or np.array_equal(kth, rkth)


@pytest.mark.parametrize("B,n_q,L,k,seed", [
    (1, 1, 4096, 256, 0), (3, 2, 1001, 64, 1), (2, 1, 9, 16, 2), (4, 1, 65536, 2048, 3),
    (2, 2, 131072, 2048, 4), (1, 1, 200003, 2048, 5), (6, 1, 2048, 2048, 6), (2, 1, 5000, 1, 7),
])
def test_topk_random(B, n_q, L, k, seed):
    g = np.random.default_rng(seed)
    s = (g.standard_normal((B, n_q, L)) * 30 + 140).astype(np.float32)
    ctx = g.integers(max(1, L // 2), L + 1, size=B)
    ctx[0] = L
    check(s, ctx, k)


@pytest.mark.parametrize("seed", range(4))
def test_topk_forced_ties(seed):
    g = np.random.default_rng(10 + seed)
    B, n_q, L = 3, 2, 3000
    k = int(g.integers(1, 600))
    s = g.integers(-3, 4, size=(B, n_q, L)).astype(np.float32) * np.float32(0.25)
    ctx = np.array([L, int(g.integers(1, L)), int(g.integers(1, k + 3))])
    check(s, ctx, k)


def test_topk_signed_zero_negative_and_extremes():
    L = 4000
    s = np.zeros((2, 1, L), np.float32)
    s[0, 0, ::2] = -0.0
    s[0, 0, 5] = np.float32(-1e-30)
    s[0, 0, 7] = np.float32(3.4e38)
    s[1, 0] = -np.abs(np.random.default_rng(3).standard_normal(L).astype(np.float32)) - 1.0
    s[1, 0, 100:200] = -np.inf
    check(s, [L, L], 1500)


def test_topk_degenerate_rows():
    s = np.random.default_rng(4).standard_normal((4, 1, 300)).astype(np.float32)
    check(s, [0, 1, 299, 300], 300)   # empty, single, short of k, exactly k
    sel, kth = gpu_topk(s, [0, 1, 5, 300], 8)
    assert list(sel[0, 0]) == [-1] * 8 and kth[0, 0] == -np.inf
    assert list(sel[1, 0]) == [0] + [-1] * 7


def test_topk_massive_ties_and_clustered_rows():
    """Threshold bins with more than a thousand keys: a row of three values (exact bins,
    ties at the k-th value decided by index) and a row whose keys crowd into one bin
    between two far outliers (more radix passes)."""
    L = 20000
    g = np.random.default_rng(8)
    s = np.empty((3, 1, L), np.float32)
    s[0, 0] = g.integers(0, 3, size=L).astype(np.float32)
    s[1, 0] = (1.0 + 1e-3 * g.standard_normal(L)).astype(np.float32)
    s[1, 0, 17] = np.float32(1e30)
    s[1, 0, 18] = np.float32(-1e30)
    s[2, 0] = np.float32(5.0)
    check(s, [L, L, L], 2048)
    check(s, [L, L - 3, 4097], 4096)
