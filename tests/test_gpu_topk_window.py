"""The decode step's top-k starts from score histograms the indexer fills over a window
of score keys chosen from each row's previous step (just below its k-th key up to its
largest).  Any window is exact -- the bins are ordered like the keys -- and a window
that misses must send the top-k to its full path.  These cases force every branch and
check the selection bit-exact against the oracle's top-k on the GPU's own scores, and
the recall (out_slot, metadata, pool bytes) against the oracle's recall on the GPU's
selection:
  - the first step (no window yet), then steps whose threshold lies in the window;
  - every score shrunk 4x (the k-th key falls below the window);
  - every score grown 4x (all keys clamp into the window's top bin, too many to resolve);
  - rows of equal keys (the threshold bin holds far more than the candidate buffer);
  - more score rows (request x query) than the workspace keeps histograms for.
After every step the workspace's histograms are back to zero and the rows that have
scores carry a valid window."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_kv_fp8_gb300 as echo
from helpers import Case, dev

pytestmark = pytest.mark.gpu

SEL_BINS, SEL_ROWS = 2048, 64


def _window_views(ws: echo.Workspace):
    """The selection histograms [64][2048] and windows [64][4] inside a workspace: the
    scratch layout puts 256-byte-aligned int32 arrays in this order: slot claims [n_g],
    nine per-entry arrays [max_rows], age histograms [4][4096], per-CTA counts [1024][4],
    global words [16], results [16], then the selection histograms and their windows."""
    a = lambda n: (n * 4 + 255) // 256 * 256
    off = (ws.c.base - ws.buf.data_ptr()) + a(ws.c.n_g) + 9 * a(ws.c.max_rows) + a(4 * 4096) + a(1024 * 4) + \
        a(16) + a(16)
    hist = ws.buf[off:off + SEL_ROWS * SEL_BINS * 4].view(torch.int32).view(SEL_ROWS, SEL_BINS)
    off2 = off + a(SEL_ROWS * SEL_BINS)
    hint = ws.buf[off2:off2 + SEL_ROWS * 16].view(torch.int32).view(SEL_ROWS, 4)
    return hist, hint


class Runner:
    def __init__(self, c: Case):
        self.c = c
        self.out = echo.StepBuffers(c.B, c.n_q, c.L_max, c.k)
        self.w = c.w.clone()
        self.clock = torch.tensor([c.clock], dtype=torch.int32, device="cuda")
        self.args = echo.make_step_args(c.pool, c.ws, c.q, self.w, c.k_index, c.ctx, c.r2h_t, c.k, self.out,
                                        clock_dev=self.clock, advance_clock=True)
        self.t = 0

    def step(self, w_scale=1.0):
        c = self.c
        self.w.copy_(c.w * w_scale)
        self.out.dev_status.zero_()
        echo.echo_decode_step(self.args)
        torch.cuda.synchronize()
        scores = self.out.scores.cpu().numpy()
        sel, kth = self.out.sel.cpu().numpy(), self.out.kth.cpu().numpy()
        sel_o, kth_o = oracle.select_topk(scores, c.inp.ctx_len, c.k)
        assert np.array_equal(sel, sel_o), f"step {self.t}: selection differs from the oracle's top-k"
        assert np.array_equal(kth, kth_o), f"step {self.t}: k-th score differs"
        out_o, status_o = c.orc_pool.prefetch_recall(sel, c.r2h, c.clock + self.t)
        assert np.array_equal(self.out.out_slot.cpu().numpy(), out_o), f"step {self.t}: out_slot differs"
        assert int(self.out.dev_status.item()) == status_o
        c.assert_pool_equal(c.orc_pool, f"step {self.t}")
        hist, hint = _window_views(c.ws)
        assert int(hist.abs().sum()) == 0, f"step {self.t}: selection histograms not back to zero"
        rows = min(c.B * c.n_q, SEL_ROWS)
        h = hint[:rows].cpu().numpy()
        assert np.all(h[:, 2] == 1), f"step {self.t}: rows without a window"
        assert np.all(h[:, 1] >= 0) and np.all(h[:, 1] <= 21)
        self.t += 1
        return sel


def test_window_hit_shrink_and_grow():
    c = Case(4, 1, 30000, 30000, 3000, 2900, clock=100, seed=61, k=512)
    r = Runner(c)
    r.step()              # no window yet: the full path, which sets the windows
    r.step()              # same scores: the threshold bin comes from the histogram
    r.step(0.25)          # every score / 4: the k-th key lies below the window
    r.step(0.25)          # the windows followed: histogram path again
    r.step(1.0)           # every score x 4: every key above the window, one overfull bin
    r.step(1.0)


def test_equal_keys_overflow_the_threshold_bin():
    c = Case(2, 1, 20000, 20000, 3000, 2900, clock=100, seed=62, k=700)
    kI = c.inp.k_index.copy()
    kI[:, 300:, :] = kI[:, :1, :]            # all but 300 tokens of each request share one key
    c.inp.k_index[...] = kI
    c.k_index.copy_(dev(kI))
    r = Runner(c)
    for _ in range(3):
        r.step()


def test_rows_beyond_the_histogram_rows():
    # 33 requests x 2 query tokens = 66 score rows: rows 64 and 65 have no histogram
    c = Case(33, 2, 4096, 4096, 40000, 30000, clock=100, seed=63, k=128)
    r = Runner(c)
    for s in (1.0, 1.0, 0.5, 0.5):
        r.step(s)
