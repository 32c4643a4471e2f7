"""Pins of the oracle's cache manager at block granularity (no GPU).

The ECHO review (marsggbo.github.io, "OSDI'26 | ECHO", section 8) notes that the
cache manager carries over to block-level sparsity by making the metadata coarser
and adding the GQA KV-head dimension.  Here a pool row is one block of tokens of one
KV head and a selection row is one (request, KV head) pair.  The cache manager's
decisions (hits, misses, victims, slots) depend only on the metadata and the
selection, never on what a row holds: the same calls on pools whose rows differ only
in length must give the same metadata and out_slot, and every resident slot must
hold exactly its host row's bytes whatever the length.
"""
import numpy as np
import pytest

import oracle
from sparse_attention_kv_fp8_gb300 import workload as wl


def run_sequence(row_elems, seed, rows=6, n_blocks=64, k=8, n_g=60, steps=4):
    n_h = rows * n_blocks
    host = wl.block_kv_pool(n_h, row_elems, seed)
    r2h = wl.req_to_host(rows, n_blocks)
    # a third of the slots hold random blocks with older clocks
    res = wl.random_resident_rows(n_h, n_g // 3, seed)
    st = wl.resident_pool(n_g, n_h, res, wl.random_clocks(res.size, 50, seed), seed)
    P = oracle.Pool.from_state(st, host)
    ctx = np.full(rows, n_blocks, np.int32)
    outs = []
    for t, sc in enumerate(wl.block_scores(rows, n_blocks, seed, steps, 0.8)):
        sel, _ = oracle.select_topk(sc, ctx, k)
        out, status = P.prefetch_recall(sel, r2h, 50 + t)
        outs.append((sel, out, status, P.metadata()))
        # guaranteed recall: every selected block is resident, with its host bytes
        assert np.all(out >= 0)
        assert np.array_equal(P.gpu_kv[out.reshape(-1)], host[r2h[np.repeat(np.arange(rows), k), sel.reshape(-1)]])
    occ = np.nonzero(P.GPUTokenFree == 0)[0]
    assert np.array_equal(P.gpu_kv[occ], host[P.GPUTokenToHost[occ]])
    return outs


def test_metadata_and_slots_do_not_depend_on_the_row_length():
    ref = run_sequence(576, 3)
    for R in (8, 1000, wl.block_row_elems()):
        got = run_sequence(R, 3)
        for (s0, o0, st0, m0), (s1, o1, st1, m1) in zip(ref, got):
            assert np.array_equal(s0, s1) and np.array_equal(o0, o1) and st0 == st1
            for key in m0:
                assert np.array_equal(m0[key], m1[key]), (R, key)


def test_kv_heads_fold_into_the_request_dimension():
    """Two KV heads of one request select their own blocks: the folded call treats
    them as two requests with disjoint host rows; the same selections made as two
    separate one-head calls (same order, same clock) give the same slots and pool
    (all but GPUIndicesBuffer, which lists the slots of the last call alone)."""
    rows, n_blocks, k, n_g, R = 2, 32, 6, 20, 64
    host = wl.block_kv_pool(rows * n_blocks, R, 5)
    r2h = wl.req_to_host(rows, n_blocks)
    sc = wl.block_scores(rows, n_blocks, 5, 1, 0.0)[0]
    sel, _ = oracle.select_topk(sc, np.full(rows, n_blocks, np.int32), k)
    A = oracle.Pool.empty(n_g, rows * n_blocks, host.copy(), row_elems=R)
    out_a, _ = A.prefetch_recall(sel, r2h, 7)
    Bp = oracle.Pool.empty(n_g, rows * n_blocks, host.copy(), row_elems=R)
    out_b = np.concatenate([Bp.prefetch_recall(sel[h:h + 1], r2h[h:h + 1], 7)[0] for h in range(rows)])
    assert np.array_equal(out_a, out_b)
    for key, v in A.metadata().items():
        if key not in ("idxbuf", "idx_count"):
            assert np.array_equal(v, Bp.metadata()[key]), key
    assert len(set(out_a.reshape(-1).tolist())) == rows * k          # no slot shared between heads


@pytest.mark.parametrize("R", [8, 4096])
def test_append_writes_whole_block_rows(R):
    rows, n_blocks, n_g = 3, 16, 10
    host = wl.block_kv_pool(rows * n_blocks, R, 9)
    r2h = wl.req_to_host(rows, n_blocks)
    P = oracle.Pool.empty(n_g, rows * n_blocks, host.copy(), row_elems=R)
    kI = np.zeros((rows, n_blocks, 128), np.uint8)
    ctx = np.array([0, 5, 15], np.int32)
    new = wl.block_kv_pool(rows, R, 10)
    new_k = np.arange(rows * 128, dtype=np.uint8).reshape(rows, 128)
    P.append(kI, ctx, r2h, new, new_k, 3)
    for b, p in enumerate((0, 5, 15)):
        h = r2h[b, p]
        assert np.array_equal(P.host_kv[h], new[b])
        assert np.array_equal(P.gpu_kv[P.HostTokenToGPU[h]], new[b])
    assert list(ctx) == [1, 6, 16]
