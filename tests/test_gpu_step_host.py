"""The host-input forms of the decode step against the device-input call, step after
step on identical layers: echo_decode_step_host (q and w copied from pinned host
memory, in one copy when w follows q in both buffers, else two) and the library's own
step graph (echo_step_graph_*), with out_slot and the status word written straight into
pinned host memory and read on the host once the call has waited.  Acceptance: every
output, the pool's metadata and bytes, the EMA and the device clock bit-identical to
echo_decode_step on the same inputs."""
import numpy as np
import pytest
import torch

import sparse_attention_kv_fp8_gb300 as echo
from helpers import Case
from test_gpu_step import StepRunner, step_inputs

pytestmark = pytest.mark.gpu

B, N_Q, L, CTX, K, N_G, RES = 3, 1, 5000, 4990, 300, 2000, 1900


class HostRunner:
    """The same layer, fed from pinned host buffers.  packed: q and w side by side in one
    pinned buffer and one device buffer (one copy per step)."""

    def __init__(self, c: Case, append: bool, packed: bool):
        self.c = c
        qb, wb = B * N_Q * 64 * 128, B * N_Q * 64 * 4
        if packed:
            self.qw_host = torch.empty(qb + wb, dtype=torch.uint8, pin_memory=True)
            self.qw_dev = torch.empty(qb + wb, dtype=torch.uint8, device="cuda")
            self.q_host = self.qw_host[:qb].view(B, N_Q, 64, 128)
            self.w_host = self.qw_host[qb:].view(torch.float32).view(B, N_Q, 64)
            q_dev = self.qw_dev[:qb].view(B, N_Q, 64, 128)
            w_dev = self.qw_dev[qb:].view(torch.float32).view(B, N_Q, 64)
        else:
            self.q_host = torch.empty((B, N_Q, 64, 128), dtype=torch.uint8, pin_memory=True)
            self.w_host = torch.empty((B, N_Q, 64), dtype=torch.float32, pin_memory=True)
            q_dev = torch.empty((B, N_Q, 64, 128), dtype=torch.uint8, device="cuda")
            w_dev = torch.empty((B, N_Q, 64), dtype=torch.float32, device="cuda")
        self.w_host.copy_(c.w.cpu())
        self.out = echo.StepBuffers(B, N_Q, L, K)
        self.res_host = torch.zeros(B * N_Q * K + 1, dtype=torch.int32, pin_memory=True)
        self.out.out_slot = self.res_host[:B * N_Q * K].view(B, N_Q, K)
        self.out.dev_status = self.res_host[B * N_Q * K:]
        self.s_hat = torch.full((B, N_Q), float("inf"), dtype=torch.float32, device="cuda")
        self.clock = torch.tensor([c.clock], dtype=torch.int32, device="cuda")
        self.new_kv = torch.zeros((B, echo.KV_ELEMS), dtype=torch.int16, device="cuda") if append else None
        self.new_ki = torch.zeros((B, echo.D_INDEX), dtype=torch.uint8, device="cuda") if append else None
        self.args = echo.make_step_args(c.pool, c.ws, q_dev, w_dev, c.k_index, c.ctx, c.r2h_t, K, self.out,
                                        stage=c.stage, s_hat=self.s_hat, new_kv=self.new_kv,
                                        new_k_index=self.new_ki, clock_dev=self.clock, advance_clock=True)

    def set_inputs(self, q, kv=None, ki=None):
        self.q_host.numpy()[...] = q
        if self.new_kv is not None:
            self.new_kv.copy_(torch.from_numpy(kv.view(np.int16)).cuda())
            self.new_ki.copy_(torch.from_numpy(ki).cuda())
        torch.cuda.synchronize()


def assert_same_layer(ref: StepRunner, cr: Case, got, cg: Case, step):
    torch.cuda.synchronize()
    for name in ("scores", "sel", "kth"):
        x, y = getattr(ref.out, name).cpu().numpy(), getattr(got.out, name).cpu().numpy()
        assert np.array_equal(x, y, equal_nan=(name == "scores")), (step, name)
    # the host read of results the kernels wrote into pinned host memory
    assert np.array_equal(ref.out.out_slot.cpu().numpy(), got.res_host[:-1].numpy().reshape(B, N_Q, K)), step
    assert int(ref.out.dev_status.item()) == int(got.res_host[-1])
    ma, mb = cr.gpu_meta(), cg.gpu_meta()
    for key in ma:
        assert np.array_equal(ma[key], mb[key]), (step, key)
    assert torch.equal(cr.pool.gpu_kv, cg.pool.gpu_kv)
    assert torch.equal(ref.s_hat, got.s_hat) and int(ref.clock.item()) == int(got.clock.item())


@pytest.mark.parametrize("packed", [True, False])
def test_host_input_step_matches_device_input_step(packed):
    cr = Case(B, N_Q, L, CTX, N_G, RES, clock=900, seed=81, k=K)
    cg = Case(B, N_Q, L, CTX, N_G, RES, clock=900, seed=81, k=K)
    ref = StepRunner(cr, s_hat0=float("inf"), append=True)
    got = HostRunner(cg, append=True, packed=packed)
    qf = cr.inp.q_float
    for step in range(4):
        qf, q, kv, ki = step_inputs(cr, step, qf)
        ref.set_inputs(q, kv, ki)
        ref.out.dev_status.zero_()
        ref.run()
        got.set_inputs(q, kv, ki)
        got.res_host[-1] = 0
        echo.echo_decode_step_host(got.args, got.q_host, got.w_host, wait=True)
        assert_same_layer(ref, cr, got, cg, step)


def test_library_step_graph_matches_eager_steps():
    cr = Case(B, N_Q, L, CTX, N_G, RES, clock=900, seed=82, k=K)
    cg = Case(B, N_Q, L, CTX, N_G, RES, clock=900, seed=82, k=K)
    ref = StepRunner(cr, s_hat0=float("inf"), append=True)
    got = HostRunner(cg, append=True, packed=True)
    g = echo.StepGraph(got.args)       # captured: nothing ran
    torch.cuda.synchronize()
    assert int(got.clock.item()) == 900 and int(got.res_host[-1]) == 0
    qf = cr.inp.q_float
    for step in range(5):
        qf, q, kv, ki = step_inputs(cr, step, qf)
        ref.set_inputs(q, kv, ki)
        ref.out.dev_status.zero_()
        ref.run()
        got.set_inputs(q, kv, ki)
        got.res_host[-1] = 0
        if step == 3:   # inputs already on the device: launch without host buffers
            got.qw_dev.copy_(got.qw_host)
            g.launch(wait=True)
        else:
            g.launch(got.q_host, got.w_host, wait=(step != 2))
            if step == 2:
                torch.cuda.synchronize()
        assert_same_layer(ref, cr, got, cg, step)
    g.close()
    g.close()   # a second close is a no-op


def test_host_input_step_two_query_tokens_without_prefetch():
    """The MTP form (two query tokens per request, each with its own top-k, one recall of
    the union) through echo_decode_step_host with separate q and w host buffers (two
    copies), prefetch off, no append: bit-identical to echo_decode_step."""
    b, nq, l, ctx, k = 4, 2, 6000, 5990, 256
    cr = Case(b, nq, l, ctx, 4000, 3500, clock=700, seed=83, k=k)
    cg = Case(b, nq, l, ctx, 4000, 3500, clock=700, seed=83, k=k)
    outs = []
    for c, host in ((cr, False), (cg, True)):
        out = echo.StepBuffers(b, nq, l, k)
        clock = torch.tensor([c.clock], dtype=torch.int32, device="cuda")
        q_dev = torch.empty((b, nq, 64, 128), dtype=torch.uint8, device="cuda")
        w_dev = torch.empty((b, nq, 64), dtype=torch.float32, device="cuda")
        q_host = torch.empty((b, nq, 64, 128), dtype=torch.uint8, pin_memory=True)
        w_host = torch.empty((b, nq, 64), dtype=torch.float32, pin_memory=True)
        args = echo.make_step_args(c.pool, c.ws, q_dev, w_dev, c.k_index, c.ctx, c.r2h_t, k, out,
                                   clock_dev=clock, advance_clock=True)
        qf = c.inp.q_float
        for step in range(3):
            qf, q, _, _ = step_inputs(c, step, qf)
            if host:
                q_host.numpy()[...] = q
                w_host.copy_(c.w.cpu())
                echo.echo_decode_step_host(args, q_host, w_host, wait=True)
            else:
                q_dev.copy_(torch.from_numpy(q).cuda())
                w_dev.copy_(c.w)
                echo.echo_decode_step(args)
                torch.cuda.synchronize()
            res = {n: getattr(out, n).cpu().numpy().copy() for n in ("scores", "sel", "kth", "out_slot")}
            outs.append((host, step, res, int(clock.item()), int(out.dev_status.item())))
    ref = [o for o in outs if not o[0]]
    got = [o for o in outs if o[0]]
    for (_, step, a, ca, sa), (_, _, g, cg_, sg) in zip(ref, got):
        for n in a:
            assert np.array_equal(a[n], g[n], equal_nan=(n == "scores")), (step, n)
        assert ca == cg_ and sa == sg, step
    ma, mb = cr.gpu_meta(), cg.gpu_meta()
    for key in ma:
        assert np.array_equal(ma[key], mb[key]), key
    assert torch.equal(cr.pool.gpu_kv, cg.pool.gpu_kv)
