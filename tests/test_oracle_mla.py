"""Pins of the oracle's sparse MLA decode (no GPU).

The ECHO review (marsggbo.github.io, "OSDI'26 | ECHO", section 2) describes MLA with
a 512-wide latent row shared by all 128 heads, and the top-k rows feeding a sparse MLA
kernel.  The oracle's attention over the selected rows is checked against PyTorch's
scaled_dot_product_attention in float64 on the gathered rows (an independent library
routine), against closed forms (a zero query averages the rows; a single row is
returned as is), and against the invariances of the definition (order of the
selection, skipped entries)."""
import numpy as np
import torch

import oracle
from sparse_attention_kv_fp8_gb300 import workload as wl


def bf16_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def setup(seed=0, B=2, n_q=2, H=8, n_g=300, k=40):
    g = np.random.default_rng(seed)
    q = wl.mla_queries(B, n_q, seed, heads=H)
    kv = wl.bf16_encode(g.standard_normal((n_g, 576), dtype=np.float32))
    sl = np.stack([np.stack([g.choice(n_g, size=k, replace=False) for _ in range(n_q)]) for _ in range(B)])
    return q, kv, sl.astype(np.int32)


def test_matches_torch_sdpa_on_the_gathered_rows():
    q, kv, sl = setup()
    sl[0, 1, 5] = -1
    sl[1, 0, :3] = -1
    scale = 1.0 / np.sqrt(192.0)
    o, lse = oracle.sparse_mla_decode(q, kv, sl, scale)
    B, n_q, H, _ = q.shape
    for b in range(B):
        for j in range(n_q):
            rows = sl[b, j][sl[b, j] >= 0]
            K = torch.from_numpy(bf16_to_f64(kv[rows]))
            Q = torch.from_numpy(bf16_to_f64(q[b, j]))
            ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], K[None, :, :512], scale=scale)[0]
            assert np.allclose(o[b, j], ref.numpy(), rtol=1e-12, atol=1e-12)
            ref_lse = torch.logsumexp(scale * (Q @ K.T), dim=-1).numpy()
            assert np.allclose(lse[b, j], ref_lse, rtol=1e-12, atol=1e-12)


def test_zero_query_averages_the_rows_and_one_row_is_returned_as_is():
    q, kv, sl = setup(1, B=1, n_q=1, H=3)
    q[...] = 0
    o, lse = oracle.sparse_mla_decode(q, kv, sl, 0.1)
    rows = bf16_to_f64(kv[sl[0, 0]])
    assert np.allclose(o[0, 0], rows[:, :512].mean(axis=0)[None], rtol=0, atol=1e-12)
    assert np.allclose(lse, np.log(sl.shape[2]))
    sl1 = np.full_like(sl, -1)
    sl1[0, 0, 7] = 11
    q2, _, _ = setup(2, B=1, n_q=1, H=3)
    o, lse = oracle.sparse_mla_decode(q2, kv, sl1, 0.1)
    assert np.array_equal(o[0, 0], np.broadcast_to(bf16_to_f64(kv[11, :512]), (3, 512)))
    s = 0.1 * (bf16_to_f64(q2[0, 0]) @ bf16_to_f64(kv[11]))
    assert np.allclose(lse[0, 0], s, rtol=1e-14)


def test_order_and_skipped_entries_do_not_matter():
    q, kv, sl = setup(3)
    o, lse = oracle.sparse_mla_decode(q, kv, sl, 0.07)
    g = np.random.default_rng(3)
    sl2 = np.concatenate([sl, np.full(sl.shape[:2] + (9,), -1, np.int32)], axis=2)
    for b in range(sl2.shape[0]):
        for j in range(sl2.shape[1]):
            sl2[b, j] = g.permutation(sl2[b, j])
    o2, lse2 = oracle.sparse_mla_decode(q, kv, sl2, 0.07)
    assert np.allclose(o, o2, rtol=1e-12, atol=1e-13) and np.allclose(lse, lse2, rtol=1e-12)


def test_no_selected_row_gives_zero_and_minus_inf():
    q, kv, sl = setup(4, B=1, n_q=1, H=2)
    o, lse = oracle.sparse_mla_decode(q, kv, np.full_like(sl, -1), 0.1)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
