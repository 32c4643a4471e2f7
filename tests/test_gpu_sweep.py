"""Corners of the sweep workload (batch 1-32 x context 16K-128K x hit rate 0.5-0.99,
k = 2048, GPU pool 200K slots, host pool B*L rows pinned): two decode steps each, the
second with step-correlated queries (the calibrated overlap sets the hit rate) and the
prefetch driven by the EMA of the first.

Per step: out_slot, the metadata arrays, counters, the recall's statistics (so the hit
rate) and the bytes of every occupied slot bit-exact against the oracle's recall on the
GPU's selection (every 16-byte vector of every host row is distinct); the selection bit-exact against the oracle's
top-k on the GPU's scores (every request up to B = 4, three sampled beyond); one
request's scores within 1e-3 of the oracle's; the EMA bit-exact."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import assert_recall_stats_equal, assert_scores_close, dev, stamp_host_rows

pytestmark = pytest.mark.gpu

K, N_G, T0 = 2048, 200_000, 3000
HERE = os.path.dirname(os.path.abspath(__file__))


def rho_for(L, overlap):
    pts = json.load(open(os.path.join(HERE, "golden", "rho_calibration.json")))["points"]
    return next(p["rho"] for p in pts if p["L"] == L and abs(p["target_overlap"] - overlap) < 1e-9)


@pytest.mark.parametrize("B,L,overlap", [(1, 16384, 0.5), (2, 32768, 0.9), (16, 65536, 0.7), (32, 131072, 0.99),
                                         (8, 131072, 0.5), (32, 16384, 0.7)])
def test_sweep_corner_two_steps(B, L, overlap):
    seed = 90 + B
    g = np.random.default_rng(seed)
    rho = rho_for(L, overlap)
    inp = wl.indexer_inputs(B, 1, 1, 1, seed)               # q, w (keys below)
    base = wl.fp8_normal(wl.rng(seed, 9), (L, echo.D_INDEX))
    k_index = np.empty((B, L, echo.D_INDEX), np.uint8)
    for b in range(B):                                       # each request: the base keys permuted
        k_index[b] = base[g.permutation(L)]
    ctx = np.full(B, L, np.int32)
    n_h = B * L
    r2h = wl.req_to_host(B, L)
    host_t = torch.empty((n_h, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    hv = host_t.numpy().view(np.uint16)
    stamp_host_rows(hv)
    n_res = min(N_G, n_h // 2)
    st = wl.resident_pool(N_G, n_h, wl.random_resident_rows(n_h, n_res, seed), wl.random_clocks(n_res, T0, seed),
                          seed)
    pool = echo.Pool(N_G, host_t)
    pool.load_state(st)
    orc = oracle.Pool.from_state(st, hv)
    ws = echo.Workspace(N_G, B * K)
    stage = echo.Stage(B, (L + 15) // 16, 16)
    out = echo.StepBuffers(B, 1, L, K)
    stats = echo.Stats()
    s_hat = torch.full((B, 1), float("inf"), dtype=torch.float32, device="cuda")
    s_hat_o = np.full((B, 1), np.inf, np.float32)
    q_buf = dev(inp.q)
    k_t, ctx_t, r2h_t, w_t = dev(k_index), dev(ctx), dev(r2h), dev(inp.w)
    args = echo.make_step_args(pool, ws, q_buf, w_t, k_t, ctx_t, r2h_t, K, out, stage=stage, s_hat=s_hat,
                               clock=T0, stats=stats)
    qf, q = inp.q_float, inp.q
    for step in range(2):
        if step:
            qf, q = wl.next_query(qf, rho, seed, step)
            q_buf.copy_(dev(q))
            args = echo.make_step_args(pool, ws, q_buf, w_t, k_t, ctx_t, r2h_t, K, out, stage=stage, s_hat=s_hat,
                                       clock=T0 + step, stats=stats)
        out.dev_status.zero_()
        before = stats.as_dict()
        echo.echo_decode_step(args)
        torch.cuda.synchronize()
        scores_g, sel, kth = out.scores.cpu().numpy(), out.sel.cpu().numpy(), out.kth.cpu().numpy()
        for b in (range(B) if B <= 4 else (0, B // 2, B - 1)):
            sel_o, kth_o = oracle.select_topk(scores_g[b:b + 1], ctx[b:b + 1], K)
            assert np.array_equal(sel[b:b + 1], sel_o) and np.array_equal(kth[b:b + 1], kth_o), (step, b)
        b = step % B
        ref = oracle.indexer_score(q[b:b + 1], inp.w[b:b + 1], k_index[b:b + 1], ctx[b:b + 1])
        assert_scores_close(scores_g[b, 0], ref[0, 0], f"step {step} scores")
        ostats = oracle.Stats()
        out_o, rs = orc.prefetch_recall(sel, r2h, T0 + step, stats=ostats)
        assert np.array_equal(out.out_slot.cpu().numpy(), out_o), f"step {step}: out_slot differs"
        assert (int(out.dev_status.item()) & ~echo.DEV_PREFETCH_CAP_HIT) == rs
        m, o = pool.metadata(), orc.metadata()
        for key in ("free", "prio", "idxbuf", "to_host", "host_to_gpu", "n_free", "idx_count"):
            assert np.array_equal(m[key], o[key]), f"step {step}: {key} differs"
        occ = np.nonzero(o["free"] == 0)[0]
        gkv = pool.gpu_kv.cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv[occ], hv[o["to_host"][occ]]), f"step {step}: bytes differ"
        s_hat_o[...] = oracle.ema_update(s_hat_o, kth)
        assert np.array_equal(s_hat.cpu().numpy(), s_hat_o)
        d = stats.as_dict()
        assert_recall_stats_equal({k_: d[k_] - before[k_] for k_ in d}, ostats.as_dict(), f"step {step}")
        hit = ostats.hits / max(1, ostats.unique_rows)
        print(f"B={B} L={L} target overlap {overlap}: step {step} hit rate {hit:.3f} (= the oracle's), "
              f"staged {d['staged']}, staged used {d['staged_used']}")
