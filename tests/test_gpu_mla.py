"""Sparse MLA decode on the GPU against the oracle (fp64).

Tolerance, derived from the arithmetic: the scores are fp32 sums of exact bf16
products (relative error ~1e-6), the softmax weights p_i enter the value product
rounded to bf16 (relative error <= 2^-9 each), so for every output element
|o_gpu - o| <= 2^-9 * sum_i p_i |v_i| / sum_i p_i + fp32 rounding; the test allows
2^-8 times that sum plus 1e-5 * max|v|.  lse within 1e-4 absolute."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import dev

pytestmark = pytest.mark.gpu

SCALE = 1.0 / np.sqrt(192.0)


def bf16_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_mla(q, kv, sl, scale=SCALE, ws=None):
    B, n_q, k = sl.shape
    q_t = dev(q.view(np.int16))
    kv_t = kv if isinstance(kv, torch.Tensor) else dev(kv.view(np.int16))
    out = torch.full((B, n_q, 128, 512), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, n_q, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = ws or echo.MlaWorkspace(B, n_q, k)
    echo.echo_sparse_mla_decode(q_t, kv_t, dev(sl), scale, out, lse, ws, dev_status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), int(st.item())


def check(q, kv_np, sl, out, lse, scale=SCALE):
    o_ref, lse_ref = oracle.sparse_mla_decode(q, kv_np, sl, scale)
    B, n_q, H, _ = q.shape
    kvf = bf16_f64(kv_np)
    for b in range(B):
        for j in range(n_q):
            valid = sl[b, j][(sl[b, j] >= 0) & (sl[b, j] < kv_np.shape[0])]
            if valid.size == 0:
                assert np.all(out[b, j] == 0) and np.all(np.isneginf(lse[b, j]))
                continue
            rows = kvf[valid]
            s = scale * (bf16_f64(q[b, j]) @ rows.T)
            p = np.exp(s - lse_ref[b, j][:, None])
            bound = p @ np.abs(rows[:, :512])                      # sum_i p_i |v_i| / l (p already / l)
            tol = 2.0 ** -8 * bound + 1e-5 * np.abs(rows[:, :512]).max()
            err = np.abs(out[b, j] - o_ref[b, j])
            assert np.all(err <= tol), f"(b={b}, j={j}) max err {err.max()} vs tol {tol[err > tol][:3]}"
            assert np.allclose(lse[b, j], lse_ref[b, j], rtol=1e-6, atol=1e-4)


def pool_rows(n_g, seed):
    return wl.bf16_encode(np.random.default_rng(seed).standard_normal((n_g, 576), dtype=np.float32))


@pytest.mark.parametrize("B,n_q,k,seed", [
    (1, 1, 16, 1),        # one chunk
    (2, 1, 256, 2),       # two full splits
    (2, 2, 300, 3),       # MTP, a ragged last split (44 rows: a partial chunk)
    (3, 1, 2048, 4),      # sixteen splits
    (2, 1, 1100, 8),      # nine splits, the last of 76 rows
    (2, 2, 8192, 9),      # 64 splits per query token, 256 CTAs
])
def test_sparse_mla_matches_oracle(B, n_q, k, seed):
    n_g = max(5000, k + 1000)
    kv = pool_rows(n_g, seed)
    q = wl.mla_queries(B, n_q, seed)
    g = np.random.default_rng(seed)
    sl = np.stack([np.stack([g.choice(n_g, size=k, replace=False) for _ in range(n_q)]) for _ in range(B)])
    sl = sl.astype(np.int32)
    sl[0, 0, g.integers(0, k, size=max(1, k // 10))] = -1     # padding / unrecalled entries
    out, lse, st = run_mla(q, kv, sl)
    assert st == 0
    check(q, kv, sl, out, lse)


def test_empty_rows_and_bad_slots():
    n_g, k = 1000, 200
    kv = pool_rows(n_g, 5)
    q = wl.mla_queries(2, 1, 5)
    g = np.random.default_rng(5)
    sl = np.stack([g.choice(n_g, size=k, replace=False) for _ in range(2)])[:, None, :].astype(np.int32)
    sl[0] = -1                                   # a query with no row
    sl[1, 0, 3] = n_g + 7                        # out of range: skipped and flagged
    out, lse, st = run_mla(q, kv, sl)
    assert st == echo.DEV_BAD_INDEX
    check(q, kv, sl, out, lse)


def test_large_logits_stay_finite():
    """Scores far from zero (scale 1): the max subtraction keeps exp in range."""
    n_g, k = 600, 512
    kv = pool_rows(n_g, 6)
    q = wl.mla_queries(1, 1, 6)
    sl = np.random.default_rng(6).choice(n_g, size=k, replace=False).astype(np.int32)[None, None]
    out, lse, st = run_mla(q, kv, sl, scale=1.0)
    assert st == 0 and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    check(q, kv, sl, out, lse, scale=1.0)


def test_attention_over_a_decode_step_reads_the_host_rows():
    """The consumer end to end: a decode step's out_slot into the MLA kernel gives
    exactly the attention over the host rows of the selected tokens (the guaranteed
    recall made every one of them resident with its host bytes)."""
    from helpers import Case
    c = Case(2, 1, 3000, 2990, 1500, 1400, clock=900, seed=77, k=256)
    out = echo.StepBuffers(2, 1, 3000, 256)
    s_hat = torch.full((2, 1), float("inf"), dtype=torch.float32, device="cuda")
    clock = torch.tensor([900], dtype=torch.int32, device="cuda")
    args = echo.make_step_args(c.pool, c.ws, c.q, c.w, c.k_index, c.ctx, c.r2h_t, 256, out, stage=c.stage,
                               s_hat=s_hat, clock_dev=clock, advance_clock=True)
    echo.echo_decode_step(args)
    torch.cuda.synchronize()
    sel = out.sel.cpu().numpy()
    slots = out.out_slot.cpu().numpy()
    assert np.all(slots[sel >= 0] >= 0)
    q = wl.mla_queries(2, 1, 77)
    o, lse, st = run_mla(q, c.pool.gpu_kv, slots)
    assert st == 0
    # the oracle attends over the host rows of the selected tokens
    host = c.host_t.numpy().view(np.uint16)
    rows = np.where(sel >= 0, c.r2h[np.arange(2)[:, None, None], np.maximum(sel, 0)], -1).astype(np.int32)
    check(q, host, rows, o, lse)


def test_workspace_reused_across_calls_and_shapes():
    """One workspace, sized for the largest call, serves repeated calls of several
    shapes (more CTAs than SMs, and fewer)."""
    n_g = 6000
    kv = pool_rows(n_g, 10)
    ws = echo.MlaWorkspace(3, 2, 4096)
    g = np.random.default_rng(10)
    for rep, (B, n_q, k) in enumerate([(3, 2, 4096), (3, 2, 4096), (2, 1, 300), (3, 1, 2048), (3, 2, 4096)]):
        q = wl.mla_queries(B, n_q, 100 + rep)
        sl = np.stack([np.stack([g.choice(n_g, size=k, replace=False) for _ in range(n_q)]) for _ in range(B)])
        sl = sl.astype(np.int32)
        out, lse, st = run_mla(q, kv, sl, ws=ws)
        assert st == 0
        check(q, kv, sl, out, lse)


def test_decode_shape_sampled():
    """The bench's configuration: 8 query tokens x 2048 selected rows drawn from a
    200K-slot pool of random rows; two of the eight query tokens checked against the
    oracle element by element."""
    n_g, B, k = 200_000, 8, 2048
    kv = pool_rows(n_g, 7)
    g = np.random.default_rng(8)
    sl = np.stack([g.choice(n_g, size=k, replace=False) for _ in range(B)]).astype(np.int32)[:, None, :]
    q = wl.mla_queries(B, 1, 31)
    out, lse, st = run_mla(q, kv, sl)
    assert st == 0 and np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    for b in (0, 5):
        check(q[b:b + 1], kv, sl[b:b + 1], out[b:b + 1], lse[b:b + 1])
