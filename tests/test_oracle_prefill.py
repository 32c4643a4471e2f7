"""Pins of the oracle's inter-query (prefill) prefetch (no GPU).

The ECHO review (marsggbo.github.io, "OSDI'26 | ECHO", section 6.2) approximates a
query's top-k by a 256-bin histogram of its scores keyed by the top 8 bits, shifted by
the predicted k-th score; the top bins whose total stays within k are prefetched, and
the section's inequality bounds what the threshold bin leaves out.  The tests check
the oracle against facts that do not come from its code: the symmetry of the
order-preserving key, monotonicity, sorting (brute force), the inequality itself, the
exact case of a perfect prediction, degenerate predictions, and a hand-built chunk.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_kv_fp8_gb300 import workload as wl


def bins_of(values, s_hat=0.0):
    """Bin of each value, read back from the oracle's histogram one value at a time."""
    out = []
    for v in values:
        _, h, _ = oracle.approx_topk_bins(np.array([v], np.float32), s_hat, 0)
        out.append(int(np.nonzero(h)[0][0]))
    return np.array(out)


def test_bins_are_monotone_symmetric_and_cover_the_range():
    g = np.random.default_rng(0)
    mags = np.concatenate([[0.0, 1e-38, 1e-30, 1e-10, 1e-3, 0.25, 1.0, 3.0, 4.0, 1e3, 1e10, 3e38],
                           np.exp(g.uniform(-80, 80, 200))]).astype(np.float32)
    vals = np.sort(np.concatenate([mags, -mags]))
    b = bins_of(vals)
    assert np.all(np.diff(b) >= 0)                                  # order preserving
    pos = mags[mags > 0]
    assert np.array_equal(bins_of(-pos), 255 - bins_of(pos))        # a sign flip mirrors the bin
    assert bins_of([0.0])[0] == bins_of([-0.0])[0] == 128           # -0 folded onto +0
    assert bins_of([np.inf])[0] == 255 and bins_of([-np.inf])[0] == 0
    # a bin of positive floats spans two binary exponents: [2, 8) is one bin, [8, 32) the next
    assert bins_of([2.0])[0] == bins_of([7.99])[0] != bins_of([8.0])[0] == bins_of([31.9])[0]
    assert bins_of([1.99])[0] != bins_of([2.0])[0]
    # every bin is reachable: one float per value of the top 8 key bits
    keys = (np.arange(256, dtype=np.uint64) << 24) | 0x123456
    floats = np.where(keys >= 0x80000000, keys ^ 0x80000000, ~keys & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    finite = np.isfinite(floats)
    assert np.array_equal(bins_of(floats[finite]), np.arange(256)[finite])


@pytest.mark.parametrize("seed", range(8))
def test_threshold_bin_inequality_and_subset_of_the_exact_top_k(seed):
    g = np.random.default_rng(seed)
    L = int(g.integers(1, 3000))
    k = int(g.integers(1, 600))
    s = (g.standard_normal(L) * g.uniform(0.1, 40) + g.uniform(-5, 200)).astype(np.float32)
    if seed % 2:
        s = np.round(s)                                              # many ties
    s_hat = np.float32(g.choice([np.sort(s)[::-1][min(k, L) - 1], np.median(s), 0.0]) + g.uniform(-3, 3))
    thr, hist, n = oracle.approx_topk_bins(s, s_hat, k)
    assert hist.sum() == L
    x = (s - s_hat).astype(np.float32)
    b = bins_of(x)
    assert np.array_equal(np.bincount(b, minlength=256), hist)
    subset = np.nonzero(b > thr)[0]
    assert subset.size == n <= k
    if L > k:
        assert thr >= 0 and n > k - hist[thr]                        # section 6.2's inequality
        assert hist[thr:].sum() > k
    else:
        assert thr == -1 and n == L
    # every token of the subset is in the exact top-k: it beats every token outside it
    if 0 < n < L:
        assert s[subset].min() > s[np.setdiff1d(np.arange(L), subset)].max()


def test_a_perfect_prediction_recovers_the_exact_top_k():
    g = np.random.default_rng(3)
    s = g.permutation(np.arange(5000, dtype=np.float32) * 0.37 + 12.5)      # distinct
    k = 731
    kth = np.sort(s)[::-1][k - 1]
    thr, hist, n = oracle.approx_topk_bins(s, kth, k)
    assert n == k
    top = np.argsort(-s, kind="stable")[:k]
    assert set(np.nonzero(bins_of(s - kth) > thr)[0].tolist()) == set(top.tolist())


def test_degenerate_predictions():
    s = np.linspace(1, 2, 100).astype(np.float32)
    for s_hat in (np.inf, -np.inf):
        thr, hist, n = oracle.approx_topk_bins(s, s_hat, 10)
        assert n == 0 and hist.max() == 100                          # one bin holds everything
    thr, _, n = oracle.approx_topk_bins(s, np.inf, 100)                   # L <= k: all of it
    assert thr == -1 and n == 100
    thr, hist, n = oracle.approx_topk_bins(np.zeros(0, np.float32), 0.0, 5)
    assert thr == -1 and n == 0 and hist.sum() == 0


def test_shift_shrinks_the_threshold_bin_on_workload_scores():
    """Section 6.2's claim, on the synthetic workload's scores: shifting by a prediction
    near the k-th score leaves a much smaller threshold bin than no shift."""
    inp = wl.indexer_inputs(2, 4, 4096, 4096, seed=9)
    sc = oracle.indexer_score(inp.q, inp.w, inp.k_index, inp.ctx_len)
    k = 256
    plain, shifted = [], []
    for b in range(2):
        for j in range(4):
            row = sc[b, j][:4096 - (3 - j)]
            kth = np.sort(row)[::-1][k - 1]
            t0, h0, _ = oracle.approx_topk_bins(row, 0.0, k)
            t1, h1, n1 = oracle.approx_topk_bins(row, kth * np.float32(1.01), k)
            plain.append(h0[t0])
            shifted.append(h1[t1])
            assert n1 > 0.8 * k
    assert np.mean(shifted) < 0.05 * np.mean(plain)


def test_prefill_candidates_hand_built_chunk():
    """Two requests, a chunk of C = 3 queries in blocks of 2, k = 2, hand-chosen scores:
    block candidates are the union over the block's queries of the tokens above each
    query's threshold bin, within each query's causal length, minus resident rows."""
    B, C, L_max, k = 2, 3, 8, 2
    ctx = np.array([8, 6], np.int32)                  # query i of request b sees ctx - (C-1-i) keys
    sc = np.full((B, C, L_max), np.nan, np.float32)
    # request 0: lengths 6, 7, 8
    sc[0, 0, :6] = [1, 9, 2, 8, 0, 0]                 # top 2 with s_hat 5: tokens 1 (9) and 3 (8)
    sc[0, 1, :7] = [7, 1, 1, 1, 1, 1, 9.5]            # tokens 0 and 6
    sc[0, 2, :8] = [1, 1, 1, 1, 1, 1, 1, 20]          # token 7 alone clears its bins
    # request 1: lengths 4, 5, 6
    sc[1, 0, :4] = [5, 5, 5, 5]                       # all in one bin: nothing below k
    sc[1, 1, :5] = [6, 40, 6, 6, 6]
    sc[1, 2, :6] = [1, 2, 3, 4, 5, 90]
    s_hat = np.array([5.0, 5.0], np.float32)
    r2h = wl.req_to_host(B, L_max)
    h2g = np.full(B * L_max, oracle.INF, np.int32)
    h2g[r2h[0, 6]] = 0                                # request 0's token 6 is resident
    thr, sub, cand = oracle.prefill_candidates(sc, s_hat, ctx, k, 2, r2h, h2g)
    # the expected sets from the scores by sorting (each query's subset is its top
    # tokens that are strictly separated from the rest by a bin boundary)
    assert [c.tolist() for c in cand[0]] == [[0, 1, 3], [7]]
    assert [c.tolist() for c in cand[1]] == [[1], [4, 5]]    # x = 0 and 85 fit k = 2; x = -1 does not
    assert sub[1, 0] == 0 and sub[0, 2] == 1
    assert np.all(sub <= k)
