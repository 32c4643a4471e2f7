"""The block-level / GQA variant of the cache manager on the GPU against the oracle.

A pool row is one block of tokens of one KV head (any multiple of 8 bf16 elements);
a selection row is one (request, KV head) pair.  Recall, allocate, evict and append
must give the oracle's out_slot, status, statistics, metadata and pool bytes
exactly, for row lengths that take the latent-row copy path's place: 16 bytes, an
odd number of 16-byte pieces, and the GQA shapes (8 KB, 32 KB)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from sparse_attention_kv_fp8_gb300 import workload as wl
from helpers import dev, pinned_host_pool

pytestmark = pytest.mark.gpu


class BlockCase:
    def __init__(self, rows, n_blocks, R, n_g, n_resident, clock, seed, k):
        self.rows, self.n_blocks, self.R, self.k = rows, n_blocks, R, k
        n_h = rows * n_blocks
        self.host_np = wl.block_kv_pool(n_h, R, seed)
        self.r2h = wl.req_to_host(rows, n_blocks)
        res = wl.random_resident_rows(n_h, n_resident, seed)
        self.state = wl.resident_pool(n_g, n_h, res, wl.random_clocks(res.size, clock, seed), seed)
        self.host_t = pinned_host_pool(self.host_np)
        self.pool = echo.Pool(n_g, self.host_t)
        self.pool.load_state(self.state)
        self.ws = echo.Workspace(n_g, max(2 * rows * k, rows))
        self.ctx_np = np.full(rows, n_blocks, np.int32)
        self.ctx = dev(self.ctx_np)
        self.r2h_t = dev(self.r2h)
        self.orc = oracle.Pool.from_state(self.state, self.host_np.copy())

    def assert_equal(self, msg):
        m, o = self.pool.metadata(), self.orc.metadata()
        for key in o:
            assert np.array_equal(m[key], o[key]), f"{msg}: {key}"
        occ = np.nonzero(o["free"] == 0)[0]
        gkv = self.pool.gpu_kv.cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv[occ], self.orc.gpu_kv[occ]), f"{msg}: pool bytes"


@pytest.mark.parametrize("R", [8, 1000, 4096, wl.block_row_elems()])
def test_block_recall_matches_oracle(R):
    rows, n_blocks, k = 2 * 4, 256, 16                   # 2 requests x 4 KV heads
    c = BlockCase(rows, n_blocks, R, n_g=160, n_resident=100, clock=40, seed=R, k=k)
    for t, sc in enumerate(wl.block_scores(rows, n_blocks, R, 4, 0.7)):
        sel, _ = oracle.select_topk(sc, c.ctx_np, k)
        out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        stats, st = echo.Stats(), torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, 40 + t, out, stats=stats, dev_status=st)
        ost = oracle.Stats()
        ref, rs = c.orc.prefetch_recall(sel, c.r2h, 40 + t, stats=ost)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref), t
        assert int(st.item()) == rs
        assert stats.as_dict() == ost.as_dict()
        c.assert_equal(f"R={R} step {t}")
    assert ost.as_dict()["evicted"] > 0                  # the last steps evicted


def test_block_alloc_evict_and_append_match_oracle():
    R, rows, n_blocks = 4096, 3, 64
    c = BlockCase(rows, n_blocks, R, n_g=40, n_resident=38, clock=9, seed=11, k=4)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_pool_evict(c.pool, c.ws, dev(np.array([5], np.int32)), 9, dev_status=st)
    c.orc.evict(5, 9)
    torch.cuda.synchronize()
    c.assert_equal("evict")
    kI = np.zeros((rows, n_blocks, 128), np.uint8)
    kI_t = dev(kI)
    ctx = np.array([10, 20, 63], np.int32)
    ctx_t = dev(ctx)
    for step in range(2):
        new = wl.block_kv_pool(rows, R, 20 + step)
        new_k = np.full((rows, 128), step + 1, np.uint8)
        echo.echo_append(c.pool, c.ws, kI_t, ctx_t, c.r2h_t, dev(new.view(np.int16)), dev(new_k), 10 + step,
                         dev_status=st)
        rs = c.orc.append(kI, ctx, c.r2h, new, new_k, 10 + step, oracle.Stats())
        torch.cuda.synchronize()
        assert int(st.item()) == rs
        assert np.array_equal(ctx_t.cpu().numpy(), ctx)
        assert np.array_equal(c.host_t.numpy().view(np.uint16), c.orc.host_kv)
        c.assert_equal(f"append {step}")


def test_prefetching_calls_need_latent_rows():
    c = BlockCase(2, 64, 1024, n_g=32, n_resident=0, clock=1, seed=12, k=4)
    stage = echo.Stage(2, 8, 16)
    sel = dev(np.zeros((2, 1, 4), np.int32))
    out = torch.empty((2, 1, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(echo.EchoError, match="576"):
        echo.echo_prefetch_recall(c.pool, c.ws, sel, c.r2h_t, c.ctx, 1, out, stage=stage)


def test_block_recall_into_a_mostly_free_pool_matches_oracle():
    """40,000 slots, 500 resident: the misses (about 4,000 a step) take the lowest free
    slots, which sit in a few CTAs' slot ranges, so the recall spreads their copies of
    2,000-byte rows over the whole grid; results equal the oracle's step after step."""
    rows, n_blocks, k, R = 8, 2048, 512, 1000
    c = BlockCase(rows, n_blocks, R, n_g=40000, n_resident=500, clock=40, seed=21, k=k)
    for t, sc in enumerate(wl.block_scores(rows, n_blocks, 21, 3, 0.7)):
        sel, _ = oracle.select_topk(sc, c.ctx_np, k)
        out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        stats, st = echo.Stats(), torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, 40 + t, out, stats=stats, dev_status=st)
        ost = oracle.Stats()
        ref, rs = c.orc.prefetch_recall(sel, c.r2h, 40 + t, stats=ost)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref), t
        assert int(st.item()) == rs
        assert stats.as_dict() == ost.as_dict()
        c.assert_equal(f"step {t}")
    assert ost.as_dict()["evicted"] == 0


def test_block_recall_at_the_bench_size():
    """The bench's block probe configuration: 4 requests x 8 KV heads, 1024 blocks of
    32 KB each (1 GiB host pool), 8192 slots; a cold recall of 64 blocks per selection
    row (2048 rows into an empty pool), then steady steps of 16 blocks from a full pool.
    Rows carry a per-row pattern over every element, so any misplaced piece shows."""
    R, rows, n_blocks, n_g = wl.block_row_elems(), 4 * wl.GQA_KV_HEADS, 1024, 8192
    n_h = rows * n_blocks
    host_np = np.empty((n_h, R), np.uint16)
    cols = np.arange(R, dtype=np.uint16)[None, :]
    for r0 in range(0, n_h, 2048):                       # (row * 7919 + col) mod 2^16
        host_np[r0:r0 + 2048] = np.arange(r0, r0 + 2048, dtype=np.uint16)[:, None] * np.uint16(7919) + cols
    host_t = pinned_host_pool(host_np)
    r2h = wl.req_to_host(rows, n_blocks)
    ctx_np = np.full(rows, n_blocks, np.int32)
    pool = echo.Pool(n_g, host_t)
    echo.echo_pool_init(pool)
    ws = echo.Workspace(n_g, rows * 64)
    orc = oracle.Pool.empty(n_g, n_h, host_np, row_elems=R)
    g = np.random.default_rng(6)
    sel = np.sort(np.stack([g.choice(n_blocks, 64, replace=False) for _ in range(rows)]), axis=1)
    sel = sel.astype(np.int32)[:, None, :]
    out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    echo.echo_prefetch_recall(pool, ws, dev(sel), dev(r2h), dev(ctx_np), 10, out, dev_status=st)
    ref, rs = orc.prefetch_recall(sel, r2h, 10)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref) and int(st.item()) == rs == 0
    m, o = pool.metadata(), orc.metadata()
    for key in o:
        assert np.array_equal(m[key], o[key]), key
    slots = ref.reshape(-1)
    gkv = pool.gpu_kv[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
    assert np.array_equal(gkv, host_np[r2h[np.repeat(np.arange(rows), 64), sel.reshape(-1)]])
    # steady steps from a full pool: every miss evicts
    res = wl.random_resident_rows(n_h, n_g, 6)
    state = wl.resident_pool(n_g, n_h, res, wl.random_clocks(n_g, 100, 6), 6)
    pool.load_state(state)
    orc = oracle.Pool.from_state(state, host_np)
    for t, sc in enumerate(wl.block_scores(rows, n_blocks, 7, 3, 0.9)):
        sel, _ = oracle.select_topk(sc, ctx_np, wl.GQA_TOPK_BLOCKS)
        out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        echo.echo_prefetch_recall(pool, ws, dev(sel), dev(r2h), dev(ctx_np), 100 + t, out, dev_status=st)
        ref, rs = orc.prefetch_recall(sel, r2h, 100 + t)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref) and int(st.item()) == rs == 0
        m, o = pool.metadata(), orc.metadata()
        for key in o:
            assert np.array_equal(m[key], o[key]), (t, key)
        slots = ref.reshape(-1)
        gkv = pool.gpu_kv[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy().view(np.uint16)
        assert np.array_equal(gkv, orc.gpu_kv[slots])


def test_block_recall_exhaustion_and_repeats():
    """Block rows when the pool cannot hold every miss (POOL_EXHAUSTED, misses left
    out with out_slot -1) and with two query tokens per (request, KV head) selecting
    overlapping blocks (repeats take the slot of the block's first entry, no copy)."""
    R, rows, n_blocks, k = 2048, 3, 128, 24
    # two query tokens per selection row: the second token's blocks overlap the first's
    c = BlockCase(rows, n_blocks, R, n_g=50, n_resident=20, clock=30, seed=13, k=k)
    g = np.random.default_rng(13)
    for t in range(3):
        sc = g.standard_normal((rows, 2, n_blocks)).astype(np.float32)
        sc[:, 1] = 0.7 * sc[:, 0] + 0.3 * sc[:, 1]
        sel, _ = oracle.select_topk(sc, c.ctx_np, k)
        out = torch.empty(sel.shape, dtype=torch.int32, device="cuda")
        stats, st = echo.Stats(), torch.zeros(1, dtype=torch.int32, device="cuda")
        echo.echo_prefetch_recall(c.pool, c.ws, dev(sel), c.r2h_t, c.ctx, 30 + t, out, stats=stats, dev_status=st)
        ost = oracle.Stats()
        ref, rs = c.orc.prefetch_recall(sel, c.r2h, 30 + t, stats=ost)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), ref), t
        assert int(st.item()) == rs and rs & echo.DEV_POOL_EXHAUSTED
        assert stats.as_dict() == ost.as_dict()
        assert ost.as_dict()["unrecalled"] > 0
        c.assert_equal(f"exhaustion step {t}")


def test_unknown_stage_flags_are_rejected():
    c = BlockCase(2, 64, 576, n_g=32, n_resident=0, clock=1, seed=14, k=4)
    stage = echo.Stage(2, 8, 16)
    stage.c.flags = 2
    sel = dev(np.zeros((2, 1, 4), np.int32))
    out = torch.empty((2, 1, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(echo.EchoError, match="flags"):
        echo.echo_prefetch_recall(c.pool, c.ws, sel, c.r2h_t, c.ctx, 1, out, stage=stage)
