"""Pins of the oracle's direct-to-slot prefetch model (no GPU).

The ECHO review (marsggbo.github.io, "OSDI'26 | ECHO", section 6.1 with the pool of
section 5) has the prefetch copy rows into the GPU pool while scoring runs; read
literally, prefetched rows take real slots.  The oracle models that with a reserve:
a recall sets aside the lowest-index free slots left after its own allocation
(evicting for them like for misses), the next step's prefetch fills them, the rows
become resident, and the next recall returns what was left unused.
Each test below derives the expected pool from the definitions by brute force
(sorted lists, sets), not from the oracle's own code.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_kv_fp8_gb300 import workload as wl


def _host(n_h, seed=0):
    return wl.host_kv_pool(n_h, seed)


def check_invariants_with_reserve(P: oracle.Pool, reserve=(), bytes_too=True):
    """Every slot is free (priority -1, no row), reserved (not free, priority -2, no
    row) or occupied (a row, the maps a bijection, bytes = host bytes; a bare
    allocate moves no bytes, hence bytes_too=False after one)."""
    free = P.GPUTokenFree.astype(bool)
    res = (~free) & (P.GPUTokenPriority == oracle.RESERVED)
    occ = (~free) & ~res
    assert sorted(np.nonzero(res)[0].tolist()) == sorted(int(s) for s in reserve)
    assert np.all(P.GPUTokenPriority[free] == -1) and np.all(P.GPUTokenToHost[free] == oracle.INF)
    assert np.all(P.GPUTokenToHost[res] == oracle.INF)
    hs = P.GPUTokenToHost[occ]
    assert np.array_equal(P.HostTokenToGPU[hs], np.nonzero(occ)[0])
    assert np.sum(P.HostTokenToGPU != oracle.INF) == occ.sum()
    assert P.n_free == free.sum()
    assert np.all(P.GPUTokenPriority[occ] >= 0)
    if bytes_too:
        assert np.array_equal(P.gpu_kv[occ], P.host_kv[hs])


def _scenario(seed, B=3, L_max=200, k=24, n_g=100, resident=80, t=50):
    g = np.random.default_rng(seed)
    n_h = B * L_max
    r2h = wl.req_to_host(B, L_max)
    rows = g.choice(n_h, size=resident, replace=False)
    st = wl.resident_pool(n_g, n_h, rows, g.integers(0, t, size=resident), seed)
    P = oracle.Pool.from_state(st, _host(n_h, seed))
    scores = g.standard_normal((B, 1, L_max)).astype(np.float32)
    sel, _ = oracle.select_topk(scores, np.full(B, L_max, np.int32), k)
    return P, sel, r2h, t, g


def _expected_rows(sel, r2h):
    rows = []
    for b in range(sel.shape[0]):
        for p in sel[b].ravel():
            if p >= 0 and int(r2h[b, p]) not in rows:
                rows.append(int(r2h[b, p]))
    return rows


@pytest.mark.parametrize("seed,R", [(1, 0), (2, 7), (3, 30), (4, 200)])
def test_reserve_is_the_next_free_slots_after_the_misses(seed, R):
    """Evictions cover the misses plus R more slots (as far as evictable slots go); the
    misses take the lowest free slots, the reserve the next R; the reserve is neither
    free nor evictable."""
    P, sel, r2h, t, _ = _scenario(seed)
    before = P.metadata()
    out, status, reserve = P.prefetch_recall(sel, r2h, clock=t, reserve_cap=R)
    rows = _expected_rows(sel, r2h)
    misses = [h for h in rows if before["host_to_gpu"][h] == oracle.INF]
    hits = [h for h in rows if before["host_to_gpu"][h] != oracle.INF]
    prio = before["prio"].copy()
    prio[before["host_to_gpu"][hits]] = t
    evictable = sorted((int(prio[s]), s) for s in range(P.n_g) if not before["free"][s] and 0 <= prio[s] < t)
    need = min(max(0, len(misses) + R - before["n_free"]), len(evictable))
    victims = sorted(s for _, s in evictable[:need])
    free_now = sorted(set(np.nonzero(before["free"])[0].tolist()) | set(victims))
    assert len(free_now) >= len(misses)
    for i, h in enumerate(misses):
        assert P.HostTokenToGPU[h] == free_now[i]
    assert reserve.tolist() == free_now[len(misses):len(misses) + R]
    assert status == 0                          # a short reserve is not an exhaustion
    assert np.all(P.GPUTokenPriority[reserve] == oracle.RESERVED) and np.all(P.GPUTokenFree[reserve] == 0)
    assert P.n_free == len(free_now) - len(misses) - len(reserve)
    assert list(P.GPUIndicesBuffer[:P.idx_count]) == free_now[:len(misses)]
    check_invariants_with_reserve(P, reserve)
    # the reserve survives calls that are not in direct mode
    n_ev, _ = P.evict(P.n_g, clock=t + 1)
    assert np.all(P.GPUTokenPriority[reserve] == oracle.RESERVED)
    fresh = [h for h in range(P.n_h) if P.HostTokenToGPU[h] == oracle.INF][:P.n_free + 5]
    slots, st = P.alloc(fresh, clock=t + 2)
    assert st & oracle.POOL_EXHAUSTED and not set(slots.tolist()) & set(reserve.tolist())
    out2, _ = P.prefetch_recall(sel, r2h, clock=t + 3)
    assert np.all(P.GPUTokenPriority[reserve] == oracle.RESERVED)
    # a direct-mode call with cap 0 returns every reserved slot
    n_free = P.n_free
    _, _, r0 = P.prefetch_recall(np.full_like(sel, -1), r2h, clock=t + 4, reserve_cap=0)
    assert r0.size == 0 and P.n_free == n_free + len(reserve)
    check_invariants_with_reserve(P, (), bytes_too=False)


def test_direct_mode_with_empty_reserve_equals_the_staging_recall():
    for seed in range(3):
        P1, sel, r2h, t, _ = _scenario(10 + seed)
        P2 = oracle.Pool(*(x.copy() if isinstance(x, np.ndarray) else x
                           for x in (P1.GPUTokenFree, P1.GPUTokenPriority, P1.GPUIndicesBuffer, P1.GPUTokenToHost,
                                     P1.HostTokenToGPU, P1.gpu_kv, P1.host_kv, P1.n_free, P1.idx_count)))
        a, sa = P1.prefetch_recall(sel, r2h, clock=t)
        b, sb, res = P2.prefetch_recall(sel, r2h, clock=t, reserve_cap=0)
        assert np.array_equal(a, b) and sa == sb and res.size == 0
        for key, v in P1.metadata().items():
            assert np.array_equal(v, P2.metadata()[key]), key


def test_prefetched_rows_are_hits_and_unselected_ones_stay_resident():
    P, sel, r2h, t, g = _scenario(21, resident=60)
    _, _, reserve = P.prefetch_recall(np.full_like(sel, -1), r2h, clock=t, reserve_cap=40)
    assert reserve.size == 40
    rows = _expected_rows(sel, r2h)
    miss = [h for h in rows if P.HostTokenToGPU[h] == oracle.INF]
    unsel = [h for h in range(P.n_h) if P.HostTokenToGPU[h] == oracle.INF and h not in rows]
    pf_rows = miss[:15] + unsel[:10]                      # 15 selected, 10 wasted
    pf_slots = reserve[[3, 0, 7, 1, 9, 2, 4, 5, 6, 8, 10, 11, 12, 13, 14, 39, 38, 20, 21, 22, 23, 24, 25, 26, 27]]
    assert P.prefetch_direct(pf_slots, pf_rows, clock=t + 1) == 0
    for s, h in zip(pf_slots, pf_rows):
        assert P.HostTokenToGPU[h] == s and P.GPUTokenToHost[s] == h and P.GPUTokenPriority[s] == t + 1
        assert np.array_equal(P.gpu_kv[s], P.host_kv[h])
    st = oracle.Stats()
    unused = sorted(set(reserve.tolist()) - set(pf_slots.tolist()))
    n_free = P.n_free
    out, status, reserve2 = P.prefetch_recall(sel, r2h, clock=t + 1, staged=[pf_rows], stats=st, reserve_cap=0)
    d = st.as_dict()
    assert d["staged"] == 25 and d["staged_used"] == 15
    assert d["misses"] == len(miss) - 15 and d["hits"] == len(rows) - d["misses"]
    for h in unsel[:10]:                                  # wasted prefetches stay resident
        assert P.HostTokenToGPU[h] in pf_slots and P.GPUTokenPriority[P.HostTokenToGPU[h]] == t + 1
    assert reserve2.size == 0
    # the unused reserve went back to the free slots before the misses took theirs
    took = sorted(P.HostTokenToGPU[h] for h in miss[15:])
    free_before = sorted(set(np.nonzero(P.GPUTokenFree)[0].tolist()) | set(took))
    assert set(unused) <= set(free_before)
    assert P.n_free == n_free + len(unused) + d["evicted"] - len(took)
    check_invariants_with_reserve(P, ())
    for b in range(sel.shape[0]):
        for i, p in enumerate(sel[b, 0]):
            assert out[b, 0, i] == P.HostTokenToGPU[r2h[b, p]] >= 0


def test_invalid_prefetch_pairs_are_flagged_and_skipped():
    P, sel, r2h, t, _ = _scenario(31, resident=50)
    _, _, reserve = P.prefetch_recall(np.full_like(sel, -1), r2h, clock=t, reserve_cap=6)
    resident_row = int(P.GPUTokenToHost[np.nonzero((P.GPUTokenFree == 0) & (P.GPUTokenPriority >= 0))[0][0]])
    free_slot = int(np.nonzero(P.GPUTokenFree)[0][0])
    absent = [h for h in range(P.n_h) if P.HostTokenToGPU[h] == oracle.INF][:3]
    meta = P.metadata()
    for slots, rows in (([free_slot], [absent[0]]),          # slot not reserved
                        ([reserve[0]], [resident_row]),       # row already resident
                        ([reserve[0]], [P.n_h + 3]),          # row out of range
                        ([P.n_g], [absent[0]])):              # slot out of range
        assert P.prefetch_direct(slots, rows, clock=t) == oracle.BAD_INDEX
        for key, v in P.metadata().items():
            assert np.array_equal(v, meta[key]), key
    # a row placed twice: the second pair is skipped
    assert P.prefetch_direct([reserve[0], reserve[1]], [absent[1], absent[1]], clock=t) == oracle.BAD_INDEX
    assert P.HostTokenToGPU[absent[1]] == reserve[0] and P.GPUTokenPriority[reserve[1]] == oracle.RESERVED


def test_append_leaves_the_reserve_alone():
    B, L_max, n_g = 2, 16, 10
    n_h = B * L_max
    P = oracle.Pool.empty(n_g, n_h, _host(n_h, 5))
    kI = np.zeros((B, L_max, 128), np.uint8)
    ctx = np.array([3, 5], np.int32)
    r2h = wl.req_to_host(B, L_max)
    P.alloc(np.array([10, 11, 12, 13, 14, 15, 28, 29], np.int32), clock=1)   # slots 0..7, rows no append touches
    sel = np.full((B, 1, 4), -1, np.int32)
    _, status, reserve = P.prefetch_recall(sel, r2h, clock=2, reserve_cap=3)
    # two free slots (8, 9) and one eviction (slot 0, the lowest of the priority-1 slots)
    assert status == 0 and reserve.tolist() == [0, 8, 9] and P.n_free == 0
    kv, kn = wl.new_tokens(B, 1, 0)
    status = P.append(kI, ctx, r2h, kv, kn, clock=4)
    # the new rows evict the two oldest occupied slots (1, 2) instead of taking reserved ones
    assert status == 0 and P.HostTokenToGPU[r2h[0, 3]] == 1 and P.HostTokenToGPU[r2h[1, 5]] == 2
    check_invariants_with_reserve(P, reserve, bytes_too=False)


def test_direct_decode_steps_keep_selection_and_bytes_independent_of_prediction():
    """The lossless property in direct mode: the selection does not depend on the
    prediction, and every selected token's slot holds its host row's bytes; the pool's
    metadata may differ (unselected prefetched rows stay resident)."""
    B, L, n_g, k = 2, 512, 300, 64
    n_h = B * L
    host = _host(n_h, 6)
    inp = wl.indexer_inputs(B, 1, L, L, seed=6)
    r2h = wl.req_to_host(B, L)
    rows = wl.random_resident_rows(n_h, 200, seed=6)
    st0 = wl.resident_pool(n_g, n_h, rows, wl.random_clocks(200, 10, 6), seed=6)
    sels, metas = [], []
    for s_hat0, cap in ((-np.inf, 48), (np.inf, 48), (150.0, 48), (np.inf, None)):
        P = oracle.Pool.from_state(st0, host)
        s_hat = np.full((B, 1), s_hat0, np.float32)
        res = oracle.Reserve(cap) if cap is not None else None
        kI, ctx = inp.k_index.copy(), inp.ctx_len.copy()
        steps = []
        for step in range(3):
            q = inp.q if step == 0 else wl.next_query(inp.q_float, 0.9, 6, step)[1]
            st = oracle.Stats()
            r = oracle.decode_step(P, q, inp.w, kI, ctx, r2h, s_hat, k, clock=10 + step, stage_stride=64,
                                   reserve=res, stats=st)
            steps.append(r["sel"].copy())
            assert r["status"] & ~oracle.PREFETCH_CAP_HIT == 0
            for b in range(B):
                sel_rows = r2h[b][r["sel"][b, 0]]
                assert np.all(r["out_slot"][b, 0] == P.HostTokenToGPU[sel_rows])
                assert np.array_equal(P.gpu_kv[r["out_slot"][b, 0]], P.host_kv[sel_rows])
            if s_hat0 == -np.inf and cap:                    # every step after the first fills
                assert st.as_dict()["staged"] == (cap if step else 0)   # the reserve the last set aside
            check_invariants_with_reserve(P, res.slots if res is not None else ())
        sels.append(steps)
        metas.append(P.metadata())
    for other in sels[1:]:
        for a, b in zip(sels[0], other):
            assert np.array_equal(a, b)
    # with +inf nothing is prefetched: direct mode differs from no prefetch only by the reserve
    assert not np.array_equal(metas[0]["host_to_gpu"], metas[1]["host_to_gpu"])
