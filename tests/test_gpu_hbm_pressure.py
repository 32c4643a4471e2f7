"""The HBM-pressure / MTP workload: batch 32, context 100K, two query tokens per request,
k = 2048, a GPU pool of only 65536 slots, hit rate about 0.5, a pinned host pool of
3.2M rows.

One step's de-duplicated selection (up to 131072 rows) does not fit the pool, so the
recall runs in four sub-batches of eight requests (at most 32768 entries each), each at
its own clock: a sub-batch's rows are protected while it is recalled and become
evictable for the next one (its attention would run in between).  After every
sub-batch: out_slot, the five metadata arrays, the counters and the bytes of every
occupied slot bit-exact against the oracle run on the GPU's selection (every 16-byte
vector of every host row is distinct), and the recall's statistics equal the oracle's.  The selection
is bit-exact against the oracle's top-k on the GPU's scores (sampled requests), and one
request's scores are within 1e-3 of the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import assert_recall_stats_equal, assert_scores_close, dev, stamp_host_rows

pytestmark = pytest.mark.gpu

B, N_Q, L, K, N_G, T0, SUB = 32, 2, 100_000, 2048, 65536, 5000, 8
N_H = B * L


def test_mtp_recall_in_sub_batches_under_hbm_pressure():
    seed = 71
    g = np.random.default_rng(seed)
    inp = wl.indexer_inputs(B, N_Q, 1, 1, seed)            # q, w (keys below)
    base = wl.fp8_normal(wl.rng(seed, 9), (L, echo.D_INDEX))
    k_index = np.empty((B, L, echo.D_INDEX), np.uint8)
    for b in range(B):                                      # each request: the base keys permuted
        k_index[b] = base[g.permutation(L)]
    ctx = np.array([L - 37 * b for b in range(B)], np.int32)
    r2h = wl.req_to_host(B, L)

    q_t, w_t, k_t, ctx_t, r2h_t = dev(inp.q), dev(inp.w), dev(k_index), dev(ctx), dev(r2h)
    scores = torch.empty((B, N_Q, L), dtype=torch.float32, device="cuda")
    sel_t = torch.empty((B, N_Q, K), dtype=torch.int32, device="cuda")
    kth_t = torch.empty((B, N_Q), dtype=torch.float32, device="cuda")
    echo.echo_indexer_score(q_t, w_t, k_t, ctx_t, scores)
    echo.echo_select_topk(scores, ctx_t, K, sel_t, kth_t)
    torch.cuda.synchronize()
    scores_g, sel, kth = scores.cpu().numpy(), sel_t.cpu().numpy(), kth_t.cpu().numpy()

    # the selection: sampled requests bit-exact on the GPU's scores; one request's scores
    for b in (0, 13, 31):
        sel_o, kth_o = oracle.select_topk(scores_g[b:b + 1], ctx[b:b + 1], K)
        assert np.array_equal(sel[b:b + 1], sel_o) and np.array_equal(kth[b:b + 1], kth_o)
    ref = oracle.indexer_score(inp.q[5:6], inp.w[5:6], k_index[5:6], ctx[5:6])
    for j in range(N_Q):
        n = int(ctx[5]) - (N_Q - 1 - j)
        assert_scores_close(scores_g[5, j, :n], ref[0, j, :n], "MTP scores")

    # pool: full, holding half of the step's selected rows (hit rate ~0.5) and other rows
    rows_sel = np.unique(np.take_along_axis(np.broadcast_to(r2h[:, None, :], (B, N_Q, L)), sel, axis=2))
    keep = g.choice(rows_sel, size=min(N_G - 4096, rows_sel.size // 2), replace=False)
    others = np.setdiff1d(g.choice(N_H, size=3 * N_G, replace=False), rows_sel)[: N_G - keep.size]
    resident = np.concatenate([keep, others])
    st = wl.resident_pool(N_G, N_H, resident, wl.random_clocks(N_G, T0, seed), seed)
    # host pool: every 16-byte vector of every row distinct (row index, vector index)
    host_t = torch.empty((N_H, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    hv = host_t.numpy().view(np.uint16)
    stamp_host_rows(hv)
    pool = echo.Pool(N_G, host_t)
    pool.load_state(st)
    orc = oracle.Pool.from_state(st, hv)                    # reads the same host rows
    ws = echo.Workspace(N_G, SUB * N_Q * K)
    out = torch.full((B, N_Q, K), -7, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stats = echo.Stats()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    recalled_before = 0
    for s in range(B // SUB):
        bs = slice(s * SUB, (s + 1) * SUB)
        clock = T0 + s
        status.zero_()
        before = stats.as_dict()
        ev[0].record()
        echo.echo_prefetch_recall(pool, ws, sel_t[bs], r2h_t[bs], ctx_t[bs], clock, out[bs], stats=stats,
                                  dev_status=status)
        ev[1].record()
        torch.cuda.synchronize()
        ostats = oracle.Stats()
        out_o, rs = orc.prefetch_recall(sel[bs], r2h[bs], clock, stats=ostats)
        assert np.array_equal(out[bs].cpu().numpy(), out_o), f"sub-batch {s}: out_slot differs"
        assert int(status.item()) == rs
        m, o = pool.metadata(), orc.metadata()
        for key in ("free", "prio", "idxbuf", "to_host", "host_to_gpu", "n_free", "idx_count"):
            assert np.array_equal(m[key], o[key]), f"sub-batch {s}: {key} differs"
        occ = np.nonzero(o["free"] == 0)[0]
        gkv = pool.gpu_kv.cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv[occ], hv[o["to_host"][occ]]), f"sub-batch {s}: bytes differ"
        st_d = stats.as_dict()
        assert_recall_stats_equal({k_: st_d[k_] - before[k_] for k_ in st_d}, ostats.as_dict(), f"sub-batch {s}")
        rec = st_d["recalled"] - recalled_before
        recalled_before = st_d["recalled"]
        print(f"sub-batch {s}: recalled {rec} rows ({rec * 1152 / 1e6:.1f} MB) in "
              f"{ev[0].elapsed_time(ev[1]):.3f} ms")
    st_d = stats.as_dict()
    assert st_d["unrecalled"] == 0 and st_d["recalled"] > 0 and st_d["evicted"] > 0
    assert 0.2 < st_d["hits"] / st_d["unique_rows"] < 0.9
