"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something it does not share code with:
library routines (torch's FP8 decoding, float64 matmul), exact integer/rational
arithmetic, brute-force characterisations, the worked allocation example printed
on the ECHO review page (section 5.2, tests/golden/allocate_worked_example.json)
and invariants the page states (lossless prefetch, eviction moves no data, the
4*N_H + 13*N_G storage law).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from sparse_attention_kv_fp8_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers that are independent of the oracle
# ---------------------------------------------------------------------------

def torch_e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def e4m3_scaled_int(code: int) -> int:
    """Integer value * 2^9 of an e4m3 code, from the bit layout (exact)."""
    s, e, m = code >> 7, (code >> 3) & 15, code & 7
    v = m if e == 0 else (8 + m) << (e - 1)   # (1+m/8)*2^(e-7) * 2^9 = (8+m) * 2^(e-1)
    return -v if s else v


def f32_round(fr: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (ties to even)."""
    x = np.float32(float(fr))
    best = None
    for c in (np.nextafter(x, np.float32(-np.inf)), x, np.nextafter(x, np.float32(np.inf))):
        d = abs(Fraction(float(c)) - fr)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(c).view(np.uint32)) & 1) == 0):
            best = (d, c)
    return np.float32(best[1])


def brute_topk(scores_row: np.ndarray, L: int, k: int):
    """Selected iff fewer than k tokens beat it (higher score, or equal score and lower index)."""
    s = scores_row[:L].astype(np.float64)
    sel = []
    for p in range(L):
        beaten_by = np.sum((s > s[p]) | ((s == s[p]) & (np.arange(L) < p)))
        if beaten_by < k:
            sel.append(p)
    return sel


# ---------------------------------------------------------------------------
# FP8 decoding
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_e4m3_to_f64(codes)
    got = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_generator_e4m3_encoding_matches_torch():
    x = np.concatenate([np.random.default_rng(3).standard_normal(50000) * 4,
                        torch_e4m3_to_f64(np.arange(0, 127, dtype=np.uint8)) * 1.0001,
                        [0.0, -0.0, 448.0, 449.0, -1000.0, 2.0 ** -10, 3 * 2.0 ** -10]]).astype(np.float32)
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(wl.e4m3_encode(x), ref)
    assert np.array_equal(wl.e4m3_encode_direct(x), ref)


def test_generator_table_encoder_equals_torch_on_random_bit_patterns():
    """The table-driven encoder against torch on random finite float32 bit patterns,
    every rounding tie between e4m3 codes, and one ulp either side of each tie."""
    g = np.random.default_rng(8)
    u = g.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = u.view(np.float32)
    x = x[np.isfinite(x)]
    mids = (torch_e4m3_to_f64(np.arange(0, 126, dtype=np.uint8)) + torch_e4m3_to_f64(np.arange(1, 127, dtype=np.uint8))) / 2
    mids = mids.astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1000))])
    x = np.concatenate([x, near, -near]).astype(np.float32)
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(wl.e4m3_encode(x), ref)


# ---------------------------------------------------------------------------
# indexer score
# ---------------------------------------------------------------------------

def test_indexer_single_head_unit_weight_is_relu_of_matvec():
    """H = 1, w = 1: s[p] = ReLU(q . k_p), checked with torch float64 matmul."""
    g = np.random.default_rng(5)
    B, n_q, H, D, L = 2, 1, 1, 128, 300
    q = wl.fp8_normal(g, (B, n_q, H, D))
    k = wl.fp8_normal(g, (B, L, D))
    w = np.ones((B, n_q, H), np.float32)
    ctx = np.array([L, 177], np.int32)
    got = oracle.indexer_score(q, w, k, ctx)
    for b in range(B):
        ref = torch.relu(torch.from_numpy(torch_e4m3_to_f64(k[b])) @ torch.from_numpy(torch_e4m3_to_f64(q[b, 0, 0])))
        ref = ref.numpy().astype(np.float32)
        assert np.array_equal(got[b, 0, :ctx[b]], ref[:ctx[b]])
        assert np.all(np.isnan(got[b, 0, ctx[b]:]))   # past the context: untouched


def test_indexer_one_hot_query_gathers_columns():
    """q_h = e_{d_h} (value 1.0), w = 1: s[p] = sum_h ReLU(k_p[d_h])."""
    g = np.random.default_rng(6)
    H, D, L = 64, 128, 257
    dims = g.integers(0, D, size=H)
    q = np.zeros((1, 1, H, D), np.uint8)
    q[0, 0, np.arange(H), dims] = 0x38  # 1.0 in e4m3
    k = wl.fp8_normal(g, (1, L, D))
    got = oracle.indexer_score(q, np.ones((1, 1, H), np.float32), k, [L])[0, 0]
    kv = torch_e4m3_to_f64(k[0])
    ref = np.maximum(kv[:, dims], 0.0).sum(axis=1).astype(np.float32)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("n_q", [1, 2])
def test_indexer_exact_rational_brute_force(n_q):
    """Exact scaled-integer dot products and exact rational head sum, rounded once to
    float32: the oracle is within half an ulp (it rounds an fp64 sum)."""
    g = np.random.default_rng(7 + n_q)
    B, H, D, L = 2, 5, 16, 9
    q = wl.fp8_normal(g, (B, n_q, H, D))
    k = wl.fp8_normal(g, (B, L, D))
    w = g.random((B, n_q, H)).astype(np.float32)
    ctx = np.array([L, 6], np.int32)
    got = oracle.indexer_score(q, w, k, ctx)
    for b in range(B):
        for j in range(n_q):
            valid = ctx[b] - (n_q - 1 - j)
            for p in range(L):
                if p >= valid:
                    assert np.isnan(got[b, j, p])
                    continue
                tot = Fraction(0)
                for h in range(H):
                    dot = sum(e4m3_scaled_int(int(q[b, j, h, d])) * e4m3_scaled_int(int(k[b, p, d]))
                              for d in range(D))
                    tot += Fraction(float(w[b, j, h])) * Fraction(max(dot, 0), 2 ** 18)
                exact = f32_round(tot)
                ulp = float(np.spacing(np.float32(abs(exact)))) if exact != 0 else 2.0 ** -149
                assert abs(Fraction(float(got[b, j, p])) - tot) <= Fraction(ulp) * Fraction(1000001, 2000000)


def test_indexer_head_weight_and_sign_matter():
    """Flipping q flips which heads pass the ReLU; scaling w scales the score."""
    g = np.random.default_rng(9)
    q = wl.fp8_normal(g, (1, 1, 64, 128))
    k = wl.fp8_normal(g, (1, 64, 128))
    w = g.random((1, 1, 64)).astype(np.float32)
    s = oracle.indexer_score(q, w, k, [64])[0, 0].astype(np.float64)
    s2 = oracle.indexer_score(q, (w * 2).astype(np.float32), k, [64])[0, 0].astype(np.float64)
    assert np.allclose(s2, 2 * s, rtol=1e-6)
    sneg = oracle.indexer_score(q ^ np.uint8(0x80), w, k, [64])[0, 0].astype(np.float64)
    qd = torch_e4m3_to_f64(q[0, 0])
    kd = torch_e4m3_to_f64(k[0])
    dots = kd @ qd.T
    full = (np.abs(dots) * w[0, 0]).sum(axis=1)  # relu(x) + relu(-x) = |x|
    assert np.allclose(s + sneg, full, rtol=1e-6)


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_topk_brute_force_with_forced_ties(seed):
    g = np.random.default_rng(100 + seed)
    B, n_q, L_max = 3, 2, 64
    k = int(g.integers(1, 40))
    scores = g.integers(-4, 5, size=(B, n_q, L_max)).astype(np.float32) * np.float32(0.5)
    ctx = np.array([L_max, int(g.integers(1, L_max)), int(g.integers(1, k + 2))], np.int32)
    sel, kth = oracle.select_topk(scores, ctx, k)
    for b in range(B):
        for j in range(n_q):
            L = max(0, ctx[b] - (n_q - 1 - j))
            ref = brute_topk(scores[b, j], L, k)
            m = min(k, L)
            assert list(sel[b, j, :m]) == ref
            assert np.all(sel[b, j, m:] == -1)
            if m:
                assert kth[b, j] == scores[b, j, ref].min()
            else:
                assert kth[b, j] == -np.inf


def test_topk_invariants_random_floats():
    g = np.random.default_rng(11)
    L, k = 5000, 300
    s = g.standard_normal((1, 1, L)).astype(np.float32)
    s[0, 0, 100:120] = s[0, 0, 50]  # a block of ties
    sel, kth = oracle.select_topk(s, [L], k)
    chosen = sel[0, 0]
    assert np.all(np.diff(chosen) > 0) and chosen.size == k
    mask = np.zeros(L, bool)
    mask[chosen] = True
    assert s[0, 0, mask].min() >= s[0, 0, ~mask].max()
    assert kth[0, 0] == s[0, 0, mask].min()
    # among tokens equal to kth, the selected ones precede the unselected ones
    eq = np.nonzero(s[0, 0] == kth[0, 0])[0]
    picked = mask[eq]
    assert np.all(np.diff(picked.astype(int)) <= 0)


def test_topk_degenerate_cases():
    s = np.zeros((1, 1, 10), np.float32)
    sel, kth = oracle.select_topk(s, [10], 4)           # all equal: first k indices
    assert list(sel[0, 0]) == [0, 1, 2, 3] and kth[0, 0] == 0.0
    sel, kth = oracle.select_topk(s, [3], 4)            # L < k: everything, -1 padded
    assert list(sel[0, 0]) == [0, 1, 2, -1]
    sel, kth = oracle.select_topk(s, [0], 4)            # empty context
    assert list(sel[0, 0]) == [-1] * 4 and kth[0, 0] == -np.inf


# ---------------------------------------------------------------------------
# cache manager
# ---------------------------------------------------------------------------

def _host(n_h, seed=0):
    return wl.host_kv_pool(n_h, seed)


def check_invariants(P: oracle.Pool, bytes_too: bool = True):
    """bytes_too=False after bare allocate/evict calls: allocate only reserves slots,
    the KV copy belongs to recall and append."""
    free = P.GPUTokenFree.astype(bool)
    occ = ~free
    assert np.array_equal(free, P.GPUTokenPriority == -1)
    assert np.array_equal(free, P.GPUTokenToHost == oracle.INF)
    hs = P.GPUTokenToHost[occ]
    assert np.array_equal(P.HostTokenToGPU[hs], np.nonzero(occ)[0])           # bijection
    assert np.sum(P.HostTokenToGPU != oracle.INF) == occ.sum()
    assert P.n_free == free.sum()
    assert np.all(P.GPUIndicesBuffer[P.idx_count:] == -1)
    if bytes_too:
        assert np.array_equal(P.gpu_kv[occ], P.host_kv[hs])                    # bytes = host bytes


def test_allocate_worked_example_from_the_page():
    ex = json.load(open(os.path.join(GOLDEN, "allocate_worked_example.json")))
    P = oracle.Pool.empty(ex["n_slots"], ex["n_host"], _host(ex["n_host"]))
    assert np.all(P.GPUTokenPriority == ex["initial_priority"])
    slots, status = P.alloc(ex["host_indices"], clock=7, tickets=ex["tickets"])
    assert status == 0
    assert list(slots) == ex["expected_slots"]
    for s, h in ex["expected_gpu_token_to_host"].items():
        assert P.GPUTokenToHost[int(s)] == h
    for h, s in ex["expected_host_token_to_gpu"].items():
        assert P.HostTokenToGPU[int(h)] == s
    assert list(P.GPUIndicesBuffer) == ex["expected_indices_buffer"]
    assert P.GPUTokenPriority[1] == 7 and P.GPUTokenPriority[4] == 7
    assert np.all(P.GPUTokenPriority[[0, 2, 3, 5]] == -1)
    assert P.GPUTokenFree.tolist() == [1, 0, 1, 1, 0, 1]


def test_allocate_default_order_takes_lowest_free_slots_and_rejects_bad_rows():
    P = oracle.Pool.empty(8, 20, _host(20))
    P.alloc([5, 6], clock=1)
    P.evict(0, clock=2)
    slots, status = P.alloc([9, 9, 5, 30, 11], clock=3)
    # 9 first occurrence -> slot 2; duplicate 9, resident 5 and out-of-range 30 rejected
    assert list(slots) == [2, -1, -1, -1, 3] and status == oracle.BAD_INDEX
    assert list(P.GPUIndicesBuffer[:2]) == [2, 3] and P.idx_count == 2
    check_invariants(P, bytes_too=False)
    slots, status = P.alloc(list(range(12, 20)), clock=4)
    assert status == oracle.POOL_EXHAUSTED and (slots >= 0).sum() == 4
    assert list(slots[:4]) == [4, 5, 6, 7] and np.all(slots[4:] == -1)
    check_invariants(P, bytes_too=False)


def test_evict_takes_smallest_priority_then_slot_and_moves_no_data():
    n_g, n_h = 8, 16
    P = oracle.Pool.empty(n_g, n_h, _host(n_h, 1))
    rows = [10, 11, 12, 13, 14, 15, 3]
    clocks = [5, 2, 2, 7, 1, 9, 3]
    for r, c in zip(rows, clocks):
        P.alloc([r], clock=c)
    # slots 0..6 hold rows 10..15,3 with priorities 5 2 2 7 1 9 3; slot 7 is free
    kv_before = P.gpu_kv.copy()
    n, status = P.evict(3, clock=9)           # slot 5 (priority 9 == clock) is protected
    assert n == 3 and status == 0
    assert sorted(np.nonzero(P.GPUTokenFree)[0].tolist()) == [1, 2, 4, 7]
    assert list(P.GPUIndicesBuffer[:3]) == [1, 2, 4] and P.idx_count == 3
    assert all(P.HostTokenToGPU[h] == oracle.INF for h in (11, 12, 14))
    assert np.array_equal(P.gpu_kv, kv_before)   # eviction is metadata only
    n, status = P.evict(10, clock=9)          # only slots 0, 3, 6 are evictable now
    assert n == 3 and status == oracle.POOL_EXHAUSTED
    assert P.GPUTokenFree[5] == 0
    check_invariants(P, bytes_too=False)


def test_metadata_storage_law():
    """4*N_H + 13*N_G bytes; about 10 MB per layer and 610 MB for 61 layers at
    N_H = 2M, N_G = 200K (section 5.1)."""
    per_layer = oracle.metadata_bytes(2_000_000, 200_000)
    assert per_layer == 4 * 2_000_000 + 13 * 200_000
    assert abs(per_layer / 2**20 - 10) < 0.5
    assert abs(61 * per_layer / 2**20 - 610) < 0.02 * 610
    P = oracle.Pool.empty(1000, 5000, _host(5000))
    meta = P.GPUTokenFree.nbytes + P.GPUTokenPriority.nbytes + P.GPUIndicesBuffer.nbytes + \
        P.GPUTokenToHost.nbytes + P.HostTokenToGPU.nbytes
    assert meta == oracle.metadata_bytes(5000, 1000)


def _scenario(seed, B=3, n_q=1, L_max=200, k=24, n_g=100, resident=90, t=50):
    g = np.random.default_rng(seed)
    n_h = B * L_max
    host = _host(n_h, seed)
    r2h = wl.req_to_host(B, L_max)
    rows = g.choice(n_h, size=resident, replace=False)
    st = wl.resident_pool(n_g, n_h, rows, g.integers(0, t, size=resident), seed)
    P = oracle.Pool.from_state(st, host)
    scores = g.standard_normal((B, n_q, L_max)).astype(np.float32)
    ctx = g.integers(k // 2, L_max + 1, size=B).astype(np.int32)
    sel, _ = oracle.select_topk(scores, ctx, k)
    return P, sel, r2h, t


@pytest.mark.parametrize("seed,n_q", [(1, 1), (2, 2), (3, 1), (4, 2)])
def test_recall_brute_force_and_invariants(seed, n_q):
    P, sel, r2h, t = _scenario(seed, n_q=n_q, n_g=100 * n_q, resident=90 * n_q)
    before = P.metadata()
    out, status = P.prefetch_recall(sel, r2h, clock=t)
    B, _, k = sel.shape
    # brute force expectation from the definitions
    rows = []
    for b in range(B):
        for j in range(n_q):
            for p in sel[b, j]:
                if p >= 0 and r2h[b, p] not in rows:
                    rows.append(int(r2h[b, p]))
    hits = [h for h in rows if before["host_to_gpu"][h] != oracle.INF]
    misses = [h for h in rows if before["host_to_gpu"][h] == oracle.INF]
    prio = before["prio"].copy()
    prio[before["host_to_gpu"][hits]] = t
    need = max(0, len(misses) - before["n_free"])
    cand = sorted((int(prio[s]), s) for s in range(P.n_g) if not before["free"][s] and prio[s] < t)
    victims = sorted(s for _, s in cand[:need])
    free_after_evict = sorted(set(np.nonzero(before["free"])[0].tolist()) | set(victims))
    assert len(free_after_evict) >= len(misses)       # the scenario is sized to fit
    for i, h in enumerate(misses):
        assert P.HostTokenToGPU[h] == free_after_evict[i]
        assert P.GPUTokenPriority[free_after_evict[i]] == t
    assert need > 0                                      # eviction is exercised
    for h in hits:
        assert P.HostTokenToGPU[h] == before["host_to_gpu"][h]
        assert P.GPUTokenPriority[before["host_to_gpu"][h]] == t
    for s in victims:
        if s not in free_after_evict[:len(misses)]:
            assert P.GPUTokenFree[s] == 1
    assert status == 0
    # every selected row resident, out_slot points at it
    for b in range(B):
        for j in range(n_q):
            for i, p in enumerate(sel[b, j]):
                if p < 0:
                    assert out[b, j, i] == -1
                else:
                    assert out[b, j, i] == P.HostTokenToGPU[r2h[b, p]] >= 0
    assert list(P.GPUIndicesBuffer[:len(misses)]) == free_after_evict[:len(misses)]
    check_invariants(P)


def test_recall_pool_exhaustion_leaves_rows_unrecalled():
    P, sel, r2h, t = _scenario(9, B=2, k=40, n_g=50, resident=50)
    P.GPUTokenPriority[:] = np.where(P.GPUTokenFree == 0, t, -1)   # everything protected
    out, status = P.prefetch_recall(sel, r2h, clock=t)
    assert status & oracle.POOL_EXHAUSTED
    assert np.sum(out == -1) > np.sum(sel == -1)
    check_invariants(P)


def test_append_is_write_through():
    B, L_max, n_g = 2, 16, 8
    n_h = B * L_max
    host = _host(n_h, 2)
    P = oracle.Pool.empty(n_g, n_h, host)
    kI = np.zeros((B, L_max, 128), np.uint8)
    ctx = np.array([3, 5], np.int32)
    r2h = wl.req_to_host(B, L_max)
    kv, kn = wl.new_tokens(B, 1, 0)
    status = P.append(kI, ctx, r2h, kv, kn, clock=4)
    assert status == 0 and list(ctx) == [4, 6]
    for b, p in ((0, 3), (1, 5)):
        h = r2h[b, p]
        assert np.array_equal(host[h], kv[b]) and np.array_equal(kI[b, p], kn[b])
        s = P.HostTokenToGPU[h]
        assert s >= 0 and P.GPUTokenPriority[s] == 4 and np.array_equal(P.gpu_kv[s], kv[b])
    check_invariants(P)


def test_append_of_a_resident_or_repeated_row_takes_and_frees_no_slot():
    """A new token's row cannot already be resident; if the caller's state says it is
    (or two requests append the same row), the row is written through, flagged, and
    neither evicts nor allocates: only the valid appends change the pool."""
    B, L_max, n_g = 3, 16, 4
    n_h = B * L_max
    host = _host(n_h, 3)
    P = oracle.Pool.empty(n_g, n_h, host)
    r2h = wl.req_to_host(B, L_max)
    r2h[2, 7] = r2h[1, 5]                     # request 2 appends request 1's row too
    ctx = np.array([3, 5, 7], np.int32)
    # full pool, oldest first: 40, then 41 and 42, then request 0's new row (resident)
    for rows, clock in (([40], 1), ([41, 42], 2), ([r2h[0, 3]], 3)):
        got, st = P.alloc(np.array(rows, np.int32), clock=clock)
        assert st == 0
    slot0 = int(got[0])
    assert P.n_free == 0
    kI = np.zeros((B, L_max, 128), np.uint8)
    kv, kn = wl.new_tokens(B, 2, 0)
    status = P.append(kI, ctx, r2h, kv, kn, clock=5)
    assert status & oracle.BAD_INDEX and list(ctx) == [4, 6, 8]
    # only request 1's row was allocated, evicting exactly one slot (the oldest: 40's)
    assert P.HostTokenToGPU[40] == oracle.INF and P.HostTokenToGPU[r2h[0, 3]] == slot0
    s1 = P.HostTokenToGPU[r2h[1, 5]]
    assert s1 >= 0 and P.GPUTokenPriority[s1] == 5 and P.n_free == 0
    assert np.array_equal(host[r2h[0, 3]], kv[0])    # written through all the same


# ---------------------------------------------------------------------------
# EMA, prefetch, lossless
# ---------------------------------------------------------------------------

def test_ema_hand_computed_sequence():
    s = np.array([np.inf], np.float32)
    seq = []
    for x in (2.0, 4.0, -1.0, -np.inf, 0.5):
        s = oracle.ema_update(s, np.array([x], np.float32), 0.5)
        seq.append(float(s[0]))
    assert seq == [2.0, 3.0, 1.0, 1.0, 0.75]


def test_prefetch_candidates_threshold_and_residency():
    scores = np.array([[[1.0, 5.0, 3.0, 3.0, 7.0, 2.0]]], np.float32)
    r2h = np.arange(6, dtype=np.int32)[None, :]
    h2g = np.full(6, oracle.INF, np.int32)
    h2g[4] = 0                                     # token 4 is resident
    cand, cap = oracle.prefetch_candidates(scores, np.array([[3.0]], np.float32), [6], r2h, h2g,
                                           stage_stride=10, cap_div=2)
    assert list(cand[0]) == [1] and cap[0] == 3     # strict '>': 3.0 does not pass
    cand, _ = oracle.prefetch_candidates(scores, np.array([[np.inf]], np.float32), [6], r2h, h2g, 10, 2)
    assert len(cand[0]) == 0


def test_lossless_selected_set_and_pool_independent_of_prediction():
    """Section 6.1: the prediction decides only what moves early, never what is selected."""
    results = []
    B, L, n_g, k = 2, 512, 300, 64
    n_h = B * L
    host = _host(n_h, 4)
    inp = wl.indexer_inputs(B, 1, L, L, seed=4)
    r2h = wl.req_to_host(B, L)
    rows = wl.random_resident_rows(n_h, 200, seed=4)
    st0 = wl.resident_pool(n_g, n_h, rows, wl.random_clocks(200, 10, 4), seed=4)
    for s_hat0 in (-np.inf, np.inf, 150.0):
        P = oracle.Pool.from_state(st0, host)
        s_hat = np.full((B, 1), s_hat0, np.float32)
        outs = []
        for step in range(3):
            q = inp.q if step == 0 else wl.next_query(inp.q_float, 0.9, 4, step)[1]
            r = oracle.decode_step(P, q, inp.w, inp.k_index.copy(), inp.ctx_len.copy(), r2h, s_hat, k,
                                   clock=10 + step, stage_stride=64)
            outs.append((r["sel"].copy(), r["out_slot"].copy()))
        results.append((outs, P.metadata(), P.gpu_kv.copy()))
    for outs, meta, kv in results[1:]:
        for (s0, o0), (s1, o1) in zip(results[0][0], outs):
            assert np.array_equal(s0, s1) and np.array_equal(o0, o1)
        for key in meta:
            assert np.array_equal(results[0][1][key], meta[key]), key
        assert np.array_equal(results[0][2], kv)
