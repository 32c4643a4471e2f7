"""Benchmark of the ECHO decode step on one GB300 (or N replicas).

One step = one layer's decode step for a batch: FP8 lightning-indexer score with
the fused prefetch -> exact top-k -> guaranteed recall (cache manager + host->HBM
copies) -> EMA, on the DeepSeek-V3.2 decode shape: B = 8 requests, context
L = 65536, k = 2048, latent KV 576 bf16 per token, host pool 1.8M rows pinned,
GPU pool 200K slots (full at the start), consecutive-step top-k overlap 0.9.

Each step replays a CUDA graph of the whole step (inputs resident in HBM); L2 is
flushed between steps (a 256 MB write, then a 256 MB read, outside the timed
events).  Prints one JSON line (rank 0): the headline steps/s, the roofline of the
indexer, e2e through the C ABI with host buffers (host wall clock), and as extra
keys the other configurations: the DeepSeek shape at overlap 0.7 with each prefetch
mode, the sweep points, the 4-layer multi-step graph and the HBM-pressure / MTP step.
`--impl reference` times the CPU oracle instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

B, L, K_TOP, N_H, N_G = 8, 65536, 2048, 1_800_000, 200_000
CAP_DIV = 16
T0 = 1000                  # step clock at the start (pre-resident rows carry older clocks)
TARGET_OVERLAP = 0.9       # the workload's; --overlap picks 0.5, 0.7 or 0.99 instead (calibrated)


def workload_name(overlap: float) -> str:
    return ("DeepSeek-V3.2 decode shape: 1 layer, B=8, L=65536, H_index=64, d_index=128 e4m3, k=2048, "
            "latent KV 576 bf16, host pool 1.8M rows pinned, GPU pool 200K slots full at start, "
            f"consecutive top-k overlap {overlap:g}")
METRIC = "decode steps/s (indexer+select+recall, one layer)"
L2_NOTE = "L2 flushed between steps outside the timed events (256 MB write, then 256 MB read)"


def rho_for(L_: int, target: float) -> float:
    path = os.path.join(ROOT, "tests", "golden", "rho_calibration.json")
    try:
        pts = json.load(open(path))["points"]
        best = min(pts, key=lambda p: (abs(p["L"] - L_), abs(p["target_overlap"] - target)))
        if best["L"] == L_ and abs(best["target_overlap"] - target) < 1e-9:
            return float(best["rho"])
    except (OSError, KeyError, ValueError):
        pass
    return 0.995


def indexer_source_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("indexer.cu", "echo_common.cuh", "cache_common.cuh", "prefetch_rows.cuh"):
        with open(os.path.join(ROOT, "sparse_attention_kv_fp8_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def nvtx_push(name: str):
    try:
        import torch
        torch.cuda.nvtx.range_push(name)
    except Exception:  # NVTX is optional
        pass


def nvtx_pop():
    try:
        import torch
        torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons every 50 ms.  It is started
    before the timed region and waited on until its first sample is in (its start-up
    must not overlap the timed steps); `window(t0, t1)` selects the samples taken while
    the timed steps ran (wall-clock times of nvidia-smi's own timestamps)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50, busy=None):
        self.idx = gpu_index
        self.period = period_ms
        self.busy = busy  # untimed GPU work run while nvidia-smi starts: the GPU must not sit idle
        self.p = None
        self.lines = []
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.p.stdout:
            self.lines.append(line)

    def __enter__(self):
        import threading
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", str(self.period)],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except OSError:
            self.p = None
            return self
        threading.Thread(target=self._reader, daemon=True).start()
        # wait for the first sample and let nvidia-smi settle; meanwhile keep the GPU busy,
        # since steps that follow an idle stretch of a few hundred ms run slow at first
        t = time.time()
        while (not self.lines or time.time() - t < 0.3) and time.time() - t < 15.0 and self.p.poll() is None:
            if self.busy is not None:
                self.busy()
            else:
                time.sleep(0.02)
        return self

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def __exit__(self, *exc):
        if self.p is not None:
            time.sleep(2.5 * self.period / 1000.0)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        return False

    @staticmethod
    def _when(stamp: str):
        try:
            main, _, frac = stamp.strip().partition(".")
            return time.mktime(time.strptime(main, "%Y/%m/%d %H:%M:%S")) + (float("0." + frac) if frac else 0.0)
        except ValueError:
            return None

    def summary(self):
        rows = []
        for line in list(self.lines):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((self._when(f[0]), float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if r[0] is not None and self.t0 is not None
                  and self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": use[-1][2] if use else None, "reasons": sorted(reasons),
                "samples": len(use), "samples_in_timed_region": len(inside),
                "timed_region_s": (self.t1 - self.t0) if self.t0 is not None else None}


def aggregate_replicas(local_total_ms: float, steps: int, pg=None, device="cpu"):
    """Whole-job throughput of N independent replicas: every rank ran `steps` steps;
    the job took as long as the slowest rank.  Returns (steps/s over all ranks,
    ms per step of the slowest rank)."""
    import torch
    world = pg.get_world_size() if pg is not None else 1
    total = local_total_ms
    if pg is not None:
        t = torch.tensor([local_total_ms], dtype=torch.float64, device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total = float(t.item())
    return world * steps / (total / 1e3), total / steps


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def build_inputs(n_steps: int, seed: int, host_out=None, overlap: float = TARGET_OVERLAP):
    from sparse_attention_kv_fp8_gb300 import workload as wl
    inp = wl.indexer_inputs(B, 1, L, L, seed=seed)
    rho = rho_for(L, overlap)
    qs = [inp.q]
    qf = inp.q_float
    for t in range(1, n_steps):
        qf, q = wl.next_query(qf, rho, seed, t)
        qs.append(q)
    host = wl.host_kv_pool(N_H, seed, n_random=B * L, out=host_out)
    r2h = wl.req_to_host(B, L)
    rows = wl.random_resident_rows(B * L, N_G, seed)
    st = wl.resident_pool(N_G, N_H, rows, wl.random_clocks(N_G, T0, seed), seed)
    return inp, qs, host, r2h, st, rho


def config_for(args, rho):
    """The workload description both arms print (the same keys in both)."""
    return {"workload": workload_name(args.overlap), "l2": L2_NOTE, "rho": rho,
            "graph": "one CUDA graph per step",
            "prefetch": "staging area" + ("" if args.prefetch_tail else
                                          "; candidates still queued when a CTA's scoring ends are dropped"),
            "priming": "an untimed pass of the same steps on a separate copy of the pool runs first",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


def cpu_baseline_sample(inp, q, host, r2h, st, requests=1):
    """Time the oracle's decode step for `requests` of the B requests (same state)."""
    import oracle
    b_sl = slice(0, requests)
    P = oracle.Pool.from_state(st, host)
    s_hat = np.full((requests, 1), np.inf, np.float32)
    t = time.perf_counter()
    oracle.decode_step(P, q[b_sl], inp.w[b_sl], inp.k_index[b_sl], inp.ctx_len[b_sl].copy(), r2h[b_sl], s_hat,
                       K_TOP, clock=T0, stage_stride=L // CAP_DIV, cap_div=CAP_DIV)
    return time.perf_counter() - t


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    # Each timed step runs the oracle's decode step for as many of the B requests as fit
    # a budget of about 90 s for the K steps (all B when K is small, at least one), and
    # its wall time is what ms_per_step reports; value scales the time per request to
    # the batch.  Two untimed single-request steps come first.
    host = np.zeros((N_H, 576), np.uint16)
    n_w = min(args.warmup, 2)
    inp, qs, host, r2h, st, rho = build_inputs(n_w + args.steps, seed=1, host_out=host, overlap=args.overlap)
    per_req = []
    for t in range(n_w):
        per_req.append(cpu_baseline_sample(inp, qs[t], host, r2h, st, requests=1))
    req_per_step = int(max(1, min(B, 90.0 / (args.steps * max(per_req[-1] if per_req else 0.3, 1e-3)))))
    step_s = []
    for t in range(args.steps):
        step_s.append(cpu_baseline_sample(inp, qs[n_w + t], host, r2h, st, requests=req_per_step))
    per_request = float(np.sum(step_s)) / (args.steps * req_per_step)
    v = 1.0 / (per_request * B)
    sample = (f"the oracle's decode step for {req_per_step} of the {B} requests (L={L}) per timed step, "
              f"{args.steps} steps after {n_w} untimed single-request steps; value = 1 / (time per request x {B})")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": float(np.mean(step_s)) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_for(args, rho),
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_kv_fp8_gb300 as echo

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    steps = args.warmup + args.steps
    n_e2e = max(3, min(args.steps, 10))
    n_wall = args.e2e_steps
    seed = 1 + rank
    host_t = torch.empty((N_H, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    inp, qs, host_np, r2h, st, rho = build_inputs(steps + min(args.steps, 10) + 2 * n_e2e + 2 * n_wall + 3, seed,
                                                  host_out=host_t.numpy().view(np.uint16), overlap=args.overlap)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        dt = cpu_baseline_sample(inp, qs[0], host_np, r2h, st, requests=args.cpu_requests)
        per_step = dt * B / args.cpu_requests
        cpu = {"value": 1.0 / per_step, "unit": "steps/s", "cores": 1, "kind": "oracle",
               "sample": (f"the oracle's decode step for {args.cpu_requests} of the {B} requests (L={L}) of one "
                          f"step: {dt:.1f} s" + ("" if args.cpu_requests == B else
                                                 f", scaled x{B / args.cpu_requests:g} to the batch"))}

    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    pool = echo.Pool(N_G, host_t)
    pool.load_state(st)
    ws = echo.Workspace(N_G, B * K_TOP)
    stage = echo.Stage(B, L // CAP_DIV, CAP_DIV, while_scoring=not args.prefetch_tail)
    out = echo.StepBuffers(B, 1, L, K_TOP)
    stats = echo.Stats()
    q_ring = dev(np.stack(qs))                       # [steps][B][1][64][128]
    w = dev(inp.w)
    k_index = dev(inp.k_index)
    ctx = dev(inp.ctx_len)
    r2h_t = dev(r2h)
    s_hat = torch.full((B, 1), float("inf"), dtype=torch.float32, device="cuda")
    clock = torch.tensor([T0], dtype=torch.int32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_rd = torch.ones(64 << 20, dtype=torch.int32, device="cuda")

    def flush_l2():
        # write a buffer larger than L2, then read another one, so each step starts
        # with an L2 that holds none of the step's data and no dirty lines
        flush.zero_()
        torch.amax(flush_rd)

    def new_events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(echo.NUM_STAGES + 1)]
        for e in evs:
            e.record()
        return evs

    def args_for(t, events=None, q=None):
        return echo.make_step_args(pool, ws, q if q is not None else q_ring[t], w, k_index, ctx, r2h_t, K_TOP, out,
                                   stage=stage, s_hat=s_hat, clock_dev=clock, advance_clock=True, stats=stats,
                                   events=events)

    # nvidia-smi starts now and samples all along: its start-up (seconds of driver
    # queries) slowed the first timed steps when it began right before them; the
    # samples taken while the timed steps run are selected by window()
    clk = ClockSampler(local)
    clk.__enter__()
    warm_host_translations(echo, torch, host_t)
    # step 0 eagerly (first calls set kernel attributes), then ONE captured step replayed
    # for every step: each step's query is copied into the graph's input buffer before
    # the step's events (outside the timed interval).  A second capture of the same step
    # with stage events (external event nodes, about 2 us each) serves the per-stage
    # breakdown loop that follows the headline loop.
    n_stage = min(args.steps, 10)
    q_buf = torch.empty_like(q_ring[0])
    q_buf.copy_(q_ring[0])
    step_args = args_for(0, q=q_buf)
    echo.echo_decode_step(step_args)
    torch.cuda.synchronize()
    stage_events = new_events()
    stage_args = args_for(0, events=stage_events, q=q_buf)
    cap_stream = torch.cuda.Stream()

    def capture(a):
        g = torch.cuda.CUDAGraph()
        cap_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(g, stream=cap_stream):
                echo.echo_decode_step(a)
        torch.cuda.current_stream().wait_stream(cap_stream)
        return g

    g_step, g_stage = capture(step_args), capture(stage_args)
    torch.cuda.synchronize()

    def timed_loop(ts):
        st = [torch.cuda.Event(enable_timing=True) for _ in ts]
        en = [torch.cuda.Event(enable_timing=True) for _ in ts]
        # the GPU spins (untimed) while the host enqueues the first steps, so that no
        # step's events enclose a wait for the host's next launch
        torch.cuda._sleep(40_000_000)
        for i, t in enumerate(ts):
            q_buf.copy_(q_ring[t], non_blocking=True)
            flush_l2()
            st[i].record()
            g_step.replay()
            en[i].record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(st, en)]

    def stage_loop(ts):
        """whole step (with the event nodes) and each stage, synchronised after every step"""
        tot, per = [], {name: [] for name in ("append", "indexer", "topk", "recall", "ema")}
        for t in ts:
            q_buf.copy_(q_ring[t], non_blocking=True)
            flush_l2()
            g_stage.replay()
            torch.cuda.synchronize()
            tot.append(stage_events[0].elapsed_time(stage_events[-1]))
            for i, name in enumerate(per):
                per[name].append(stage_events[i].elapsed_time(stage_events[i + 1]))
        return tot, per

    timed = list(range(args.warmup, args.warmup + args.steps))

    # priming: the first timed loop of a process ran 4-6 us per step slower than any
    # later one, whichever prefetch mode it used, so an untimed pass of the same steps
    # on a separate copy of the pool runs first (the measured pool is not touched)
    prefetch_mode_leg(echo, torch, st, host_t, q_ring, w, k_index, ctx, r2h_t, flush_l2, args.warmup,
                      min(args.steps, 200), n_stage, -1, not args.prefetch_tail)
    try:
        # the warm-up steps run right before the timed ones (no idle gap between them)
        for t in range(1, args.warmup):
            q_buf.copy_(q_ring[t], non_blocking=True)
            flush_l2()
            g_step.replay()
        torch.cuda.synchronize()
        stats.t.zero_()
        out.dev_status.zero_()
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        nvtx_push("echo_timed_steps")  # lets a profiler pick out the timed steps' launches
        t_start = time.time()
        step_ms = timed_loop(timed)
        clk.window(t_start, time.time())
        nvtx_pop()
    finally:
        clk.__exit__(None, None, None)
    if pg:
        pg.barrier()
    st_vals = stats.as_dict()
    status = int(out.dev_status.item())
    staged_total_ms, stage_ms = stage_loop(list(range(steps, steps + n_stage)))
    status |= int(out.dev_status.item())
    value, ms_per_step = aggregate_replicas(float(np.sum(step_ms)), args.steps, pg, device="cuda")

    # ---- e2e: the C-ABI call with host buffers (q, w in; out_slot, status out) ----
    # the inputs travel in one copy (q and w side by side in one pinned buffer and one
    # device buffer); the kernels write the results (out_slot and status, side by side)
    # straight into pinned host memory (zero-copy: the API takes any device-accessible
    # pointer for them)
    q_bytes, w_bytes = B * 64 * 128, B * 64 * 4
    qw_host = torch.empty(q_bytes + w_bytes, dtype=torch.uint8, pin_memory=True)
    qw_dev = torch.empty(q_bytes + w_bytes, dtype=torch.uint8, device="cuda")
    q_host = qw_host[:q_bytes].view(B, 1, 64, 128)
    qw_host[q_bytes:].view(torch.float32).copy_(torch.from_numpy(inp.w.reshape(-1)))
    q_dev = qw_dev[:q_bytes].view(B, 1, 64, 128)
    w_dev = qw_dev[q_bytes:].view(torch.float32).view(B, 1, 64)
    res_host = torch.empty(B * K_TOP + 1, dtype=torch.int32, pin_memory=True)
    out_e = echo.StepBuffers(B, 1, L, K_TOP)
    res_host.zero_()
    out_e.out_slot = res_host[:B * K_TOP].view(B, 1, K_TOP)
    out_e.dev_status = res_host[B * K_TOP:]
    ea = echo.make_step_args(pool, ws, q_dev, w_dev, k_index, ctx, r2h_t, K_TOP, out_e, stage=stage, s_hat=s_hat,
                             clock_dev=clock, advance_clock=True, stats=stats)
    w_host = qw_host[q_bytes:].view(torch.float32)

    def e2e_body(wait=False):
        # the C ABI's host-input step: the copy of q and w and the step's launches in one call
        echo.echo_decode_step_host(ea, q_host, w_host, wait=wait)

    def e2e_loop(run, first):
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
        for i in range(n_e2e):
            q_host.numpy()[...] = qs[first + i]
            flush_l2()
            torch.cuda._sleep(400_000)  # untimed: the host's launch is queued before the step's events
            e_s[i].record()
            run()
            e_e[i].record()
            torch.cuda.synchronize()   # the host reads this step's out_slot and status
        return float(np.mean([s.elapsed_time(e) for s, e in zip(e_s, e_e)]))

    # direct calls, then the library's step graph (the way a serving loop runs it: the
    # step captured once, the clock on the device, the input copy issued before each launch)
    e2e_eager_ms = e2e_loop(e2e_body, steps + n_stage)
    eg = echo.StepGraph(ea)

    def e2e_graph(wait=False):
        eg.launch(q_host, w_host, wait=wait)

    q_host.numpy()[...] = qs[steps + n_stage + 2 * n_e2e]  # one untimed launch first
    e2e_graph()
    torch.cuda.synchronize()
    h2d = qw_host.numel()
    d2h = res_host.numel() * 4

    # the same calls timed by the host's wall clock: from the moment the step's inputs are
    # in pinned host memory to the moment the host holds its out_slot and status
    # (perf_counter around: the input copy, the C-ABI call or the graph launch, a stream
    # synchronisation, the host's read of the results); L2 flushed before each step
    # outside the measurement, no GPU work queued ahead
    res_np = res_host.numpy()   # one numpy view of the pinned results, made once
    got = np.empty_like(res_np)  # the host's copy of the results, reused every step

    def e2e_wall(run, first):
        ts = []
        for i in range(n_wall):
            q_host.numpy()[...] = qs[first + i]
            flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            run(wait=True)   # returns once the stream has finished the step
            np.copyto(got, res_np)
            ts.append(time.perf_counter() - t0)
        return np.array(ts) * 1e6

    wall_first = steps + n_stage + 2 * n_e2e + 1
    wall_direct = e2e_wall(e2e_body, wall_first)
    wall_graph = e2e_wall(e2e_graph, wall_first + n_wall)

    # ---- host-link denominators: pinned H2D copy (copy engine), best of 10 ----
    src = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    best = 1e9
    for _ in range(10):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        dst.copy_(src, non_blocking=True)
        a1.record()
        torch.cuda.synchronize()
        best = min(best, a0.elapsed_time(a1))
    h2d_gbs = (256 << 20) / (best * 1e-3) / 1e9
    recall_probe = recall_bandwidth_probe(echo, torch, host_t, flush_l2)
    block_probe = block_recall_probe(echo, torch, flush_l2, h2d_gbs)
    volume_probe = indexer_volume_probe(echo, torch, inp, flush_l2, hbm_peak)
    # the prefill chunk indexer (inter-query prefetch row): 1216 queries = 304 blocks of 4,
    # two full waves on 152 SMs; FP8 tensor peak = the measured bf16 peak x 2
    pre = prefill_probe(echo, torch, flush_l2, B=1, L_=32768, C=1216)
    mla = mla_probe(echo, torch, flush_l2, pool, out.out_slot, hbm_peak, float(peaks.get("bf16_tflops", 1900.0)))
    fp8_peak = 2.0 * float(peaks.get("bf16_tflops", 1900.0))
    pre["roofline"] = {"bound": "tensor", "peak": fp8_peak, "unit": "TFLOP/s",
                       "frac_scores": pre["tflops_scores"] / fp8_peak,
                       "peak_source": ("measured bf16 x 2" if "bf16_tflops" in peaks else "fallback bf16 x 2")}
    direct = off = None
    if args.reserve > 0:
        direct = prefetch_mode_leg(echo, torch, st, host_t, q_ring, w, k_index, ctx, r2h_t, flush_l2,
                                   args.warmup, args.steps, n_stage, args.reserve, not args.prefetch_tail)
        off = prefetch_mode_leg(echo, torch, st, host_t, q_ring, w, k_index, ctx, r2h_t, flush_l2,
                                args.warmup, args.steps, n_stage, 0)

    # ---- the other configurations and the hit-rate point of the DeepSeek shape ----
    extra = {}
    if not args.headline_only:
        big_rows = max(max(b_ * l_ for b_, l_, _ in SWEEP_POINTS), 32 * 100_000, 4 * 16 * (32768 + 256))
        host_big = torch.empty((big_rows, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
        n_leg = min(args.steps, 30)
        extra["deepseek_overlap_0.7"] = {
            m: decode_config_leg(echo, torch, flush_l2, host_big, B, L, 0.7, m, n_leg, 301, hbm_peak, h2d_gbs)
            for m in ("staging", "direct", "off")}
        ov = extra["deepseek_overlap_0.7"]
        extra["deepseek_overlap_0.7"]["exposed_recall_us"] = {m: ov[m]["stage_ms"]["recall"] * 1e3
                                                              for m in ("staging", "direct", "off")}
        extra["sweep"] = [decode_config_leg(echo, torch, flush_l2, host_big, b_, l_, o_, "off", n_leg, 400 + i,
                                            hbm_peak, h2d_gbs) for i, (b_, l_, o_) in enumerate(SWEEP_POINTS)]
        extra["multi_step"] = multistep_leg(echo, torch, flush_l2, host_big)
        extra["hbm_pressure_mtp"] = mtp_leg(echo, torch, flush_l2, host_big, hbm_peak, h2d_gbs)
        del host_big

    # ---- roofline of the dominant kernel (the indexer) ----
    idx_ms = float(np.mean(stage_ms["indexer"]))
    idx_bytes = B * L * 128 + B * L * 4 + B * (64 * 128 + 64 * 4)       # k_index + scores + q/w per launch
    achieved = idx_bytes / (idx_ms * 1e-3) / 1e9
    traffic = None
    prof = os.path.join(ROOT, "profiles", "indexer_traffic.json")
    if os.path.exists(prof):
        try:
            rec = json.load(open(prof))
            # counters taken from another version of the kernel do not count
            if rec.get("source_sha256") == indexer_source_sha256():
                traffic = rec.get("bytes_per_launch_full_shape")
        except (OSError, ValueError):
            traffic = None
    recalled_rows = st_vals["recalled"]
    recall_ms = float(np.mean(stage_ms["recall"]))
    hits, uniq = st_vals["hits"], max(1, st_vals["unique_rows"])
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3 x e4m3 -> f32 (indexer); int32 metadata; bf16 bytes",
        "data": "synthetic",
        "config": config_for(args, rho),
        "scored_tokens_per_s": value * B * L,
        "step_us": {"p10": float(np.percentile(step_ms, 10)) * 1e3, "p50": float(np.median(step_ms)) * 1e3,
                    "p90": float(np.percentile(step_ms, 90)) * 1e3,
                    "first_tenth_mean": float(np.mean(step_ms[:max(1, len(step_ms) // 10)])) * 1e3,
                    "last_tenth_mean": float(np.mean(step_ms[-max(1, len(step_ms) // 10):])) * 1e3},
        "hit_rate": hits / uniq,
        "recalled_rows_per_step": recalled_rows / args.steps,
        "staged_rows_per_step": st_vals["staged"] / args.steps,
        "staged_used_per_step": st_vals["staged_used"] / args.steps,
        "evicted_per_step": st_vals["evicted"] / args.steps,
        "prefill_chunk": pre,
        "sparse_mla_decode": mla,
        "block_gqa_recall": block_probe,
        "direct_to_slot": direct,
        "prefetch_off": off,
        "stage_ms": {k: float(np.mean(v)) for k, v in stage_ms.items()},
        "stage_ms_note": f"from {n_stage} further steps replayed with stage events ({float(np.mean(staged_total_ms)):.4f} ms/step with the events)",
        "recall": {"bytes_per_step": recalled_rows / args.steps * 1152, "ms": recall_ms,
                   "probe": recall_probe, "h2d_gbs_copy_engine": h2d_gbs},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic, "kernel": "indexer_kernel<1>",
                     "peak_source": peak_src, "bytes_per_launch": idx_bytes},
        "indexer_volume": volume_probe,
        "cpu_baseline": cpu,
        "e2e": {"value": 1e6 / float(np.median(wall_direct)), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": ("host wall clock (median of %d steps) from inputs in pinned host memory to results "
                        "read by the host: echo_decode_step_host through the C ABI (one copy of q and w "
                        "from one pinned buffer, the step's launches, a wait for the stream), then the "
                        "host read of out_slot and status (written by the kernels straight into pinned "
                        "host memory)" % n_wall),
                "wall_us": {"p10": float(np.percentile(wall_direct, 10)), "p50": float(np.median(wall_direct)),
                            "p90": float(np.percentile(wall_direct, 90))},
                "all_slots_valid": bool((out_e.out_slot >= 0).all().item()),
                "device": {"value": 1e3 / e2e_eager_ms, "unit": "steps/s",
                           "how": "the same calls timed by CUDA events on the stream, launches queued before "
                                  "the first event (device side only)"},
                "graph": {"value": 1e6 / float(np.median(wall_graph)), "unit": "steps/s",
                          "wall_us": {"p10": float(np.percentile(wall_graph, 10)),
                                      "p50": float(np.median(wall_graph)),
                                      "p90": float(np.percentile(wall_graph, 90))},
                          "how": "the same through the library's step graph (echo_step_graph_launch: the "
                                 "input copy, then the captured step)"}},
        **extra,
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "dev_status": status,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def prefetch_mode_leg(echo, torch, st, host_t, q_ring, w, k_index, ctx, r2h_t, flush_l2, warmup, n_timed, n_stage,
                      reserve, while_scoring=True):
    """The same steps (same start state, same queries) with another prefetch mode:
    reserve > 0, direct to slot (rows land in `reserve` slots each recall sets aside,
    instead of the staging area); reserve = 0, no prefetch at all (the whole miss set
    is recalled after the top-k); reserve < 0, the staging area again.  Whole steps
    and the per-stage split, timed as in the main loop."""
    pool = echo.Pool(N_G, host_t)
    pool.load_state(st)
    ws = echo.Workspace(N_G, B * K_TOP)
    stage = echo.Stage(B, reserve=reserve, while_scoring=while_scoring) if reserve > 0 else (
        echo.Stage(B, L // CAP_DIV, CAP_DIV, while_scoring=while_scoring) if reserve < 0 else None)
    out = echo.StepBuffers(B, 1, L, K_TOP)
    stats = echo.Stats()
    s_hat = torch.full((B, 1), float("inf"), dtype=torch.float32, device="cuda")
    clock = torch.tensor([T0], dtype=torch.int32, device="cuda")

    q_buf = torch.empty_like(q_ring[0])

    def args_for(events=None):
        return echo.make_step_args(pool, ws, q_buf, w, k_index, ctx, r2h_t, K_TOP, out, stage=stage,
                                   s_hat=s_hat, clock_dev=clock, advance_clock=True, stats=stats, events=events)

    steps = warmup + n_timed
    q_buf.copy_(q_ring[0])
    step_args = args_for()
    echo.echo_decode_step(step_args)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(echo.NUM_STAGES + 1)]
    for x in evs:
        x.record()
    stage_args = args_for(events=evs)
    cap = torch.cuda.Stream()

    def capture(a):
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                echo.echo_decode_step(a)
        torch.cuda.current_stream().wait_stream(cap)
        return g

    g_step, g_stage = capture(step_args), capture(stage_args)
    for t in range(1, warmup):
        q_buf.copy_(q_ring[t], non_blocking=True)
        flush_l2()
        g_step.replay()
    torch.cuda.synchronize()
    stats.t.zero_()
    out.dev_status.zero_()

    a_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    b_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
    torch.cuda._sleep(40_000_000)  # the host enqueues ahead while the GPU spins (untimed)
    for i, t in enumerate(range(warmup, steps)):
        q_buf.copy_(q_ring[t], non_blocking=True)
        flush_l2()
        a_ev[i].record()
        g_step.replay()
        b_ev[i].record()
    torch.cuda.synchronize()
    ms = [x.elapsed_time(y) for x, y in zip(a_ev, b_ev)]
    sv = stats.as_dict()
    status = int(out.dev_status.item())
    per_stage = {name: [] for name in ("append", "indexer", "topk", "recall", "ema")}
    for t in range(steps, steps + n_stage):
        q_buf.copy_(q_ring[t], non_blocking=True)
        flush_l2()
        g_stage.replay()
        torch.cuda.synchronize()
        for i, name in enumerate(per_stage):
            per_stage[name].append(evs[i].elapsed_time(evs[i + 1]))
    stage_ms = {name: float(np.mean(v)) for name, v in per_stage.items()}
    per = float(np.mean(ms))
    return {"mode": "direct to slot" if reserve > 0 else ("no prefetch" if reserve == 0 else "staging"),
            "reserve_slots": max(reserve, 0),
            "value": 1e3 / per, "unit": "steps/s", "ms_per_step": per,
            "step_us": {"p10": float(np.percentile(ms, 10)) * 1e3, "p50": float(np.median(ms)) * 1e3,
                        "p90": float(np.percentile(ms, 90)) * 1e3, "max": float(np.max(ms)) * 1e3},
            "hit_rate": sv["hits"] / max(1, sv["unique_rows"]),
            "recalled_rows_per_step": sv["recalled"] / n_timed,
            "prefetched_rows_per_step": sv["staged"] / n_timed,
            "prefetched_selected_per_step": sv["staged_used"] / n_timed,
            "evicted_per_step": sv["evicted"] / n_timed,
            "stage_ms": stage_ms, "dev_status": status}


# ---------------------------------------------------------------------------
# the other configurations: inputs drawn on the GPU (seeded torch generator), so that
# half-gigabyte key caches and multi-gigabyte host pools are ready in seconds; their
# content does not change the timing (the parity tests run these shapes against the
# oracle with the workload module's inputs)
# ---------------------------------------------------------------------------
def gpu_indexer_inputs(torch, B_, n_q, L_, seed, chunk=1 << 24):
    """k^I [B][L][128] e4m3, q as its pre-rounding draw [B][n_q][64][128] and w [B][n_q][64]:
    N(0,1) clamped to +-8, rounded to e4m3 (torch's conversion), w ~ U(0,1)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    k = torch.empty((B_ * L_, 128), dtype=torch.uint8, device="cuda")
    for r0 in range(0, B_ * L_, chunk // 128):
        r1 = min(B_ * L_, r0 + chunk // 128)
        k[r0:r1] = torch.randn((r1 - r0, 128), generator=g, device="cuda").clamp_(-8, 8).to(
            torch.float8_e4m3fn).view(torch.uint8)
    qf = torch.randn((B_, n_q, 64, 128), generator=g, device="cuda").clamp_(-8, 8)
    w = torch.rand((B_, n_q, 64), generator=g, device="cuda")
    return k.view(B_, L_, 128), qf, w, g


def gpu_query_ring(torch, qf, rho, n, g):
    """n step-correlated queries q_{t+1} = rho q_t + sqrt(1 - rho^2) eps (e4m3), from qf."""
    out = torch.empty((n,) + tuple(qf.shape), dtype=torch.uint8, device="cuda")
    for t in range(n):
        if t:
            qf = (rho * qf + float(np.sqrt(max(0.0, 1 - rho * rho))) *
                  torch.randn(qf.shape, generator=g, device="cuda")).clamp_(-8, 8)
        out[t] = qf.to(torch.float8_e4m3fn).view(torch.uint8)
    return out


def pool_state_for(n_g, n_h, seed, clock0=T0):
    """A pool full at the start (half the referenced rows when they fit) with clocks below
    the step clock."""
    from sparse_attention_kv_fp8_gb300 import workload as wl
    n_res = min(n_g, n_h // 2) if n_h < 2 * n_g else n_g
    return wl.resident_pool(n_g, n_h, wl.random_resident_rows(n_h, n_res, seed), wl.random_clocks(n_res, clock0, seed),
                            seed)


def replay_timed(torch, g_step, before, flush_l2, n):
    """n replays of g_step, each after before(i) and an L2 flush (outside the events);
    returns the per-step times in ms."""
    ms = []
    for i in range(n):
        before(i)
        flush_l2()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        g_step.replay()
        a1.record()
        torch.cuda.synchronize()
        ms.append(a0.elapsed_time(a1))
    return ms


def capture_graph(torch, fn):
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            fn()
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    return g


def decode_config_leg(echo, torch, flush_l2, host_big, B_, L_, overlap, mode, n_timed, seed, hbm_peak, h2d_gbs,
                      n_g=N_G, warmup=4, n_stage=5, reserve=8192):
    """One decode-step configuration (B_ requests of context L_, k = 2048, n_g GPU slots,
    host rows B_ * L_ from the shared pinned buffer) timed like the headline: one captured
    step replayed per step, L2 flushed between steps, stage times from a second capture
    with stage events.  mode: "staging", "direct" (reserve slots) or "off" (no prefetch).
    Algorithmic bytes of the indexer: B_ L_ (128 + 4) + B_ (8192 + 256); of the recall:
    1152 per recalled row, read from the host pool (all of them with the prefetch off)."""
    rho = rho_for(L_, overlap)
    k_index, qf, w, g = gpu_indexer_inputs(torch, B_, 1, L_, seed)
    steps = warmup + n_timed + n_stage
    q_ring = gpu_query_ring(torch, qf, rho, steps + 1, g)
    n_h = B_ * L_
    r2h = torch.arange(n_h, dtype=torch.int32, device="cuda").view(B_, L_)
    ctx = torch.full((B_,), L_, dtype=torch.int32, device="cuda")
    pool = echo.Pool(n_g, host_big[:n_h])
    pool.load_state(pool_state_for(n_g, n_h, seed), gpu_kv=pool.gpu_kv)
    ws = echo.Workspace(n_g, B_ * K_TOP)
    stage = (echo.Stage(B_, L_ // CAP_DIV, CAP_DIV, while_scoring=True) if mode == "staging" else
             echo.Stage(B_, reserve=reserve, while_scoring=True) if mode == "direct" else None)
    out = echo.StepBuffers(B_, 1, L_, K_TOP)
    stats = echo.Stats()
    s_hat = torch.full((B_, 1), float("inf"), dtype=torch.float32, device="cuda")
    clock = torch.tensor([T0], dtype=torch.int32, device="cuda")
    q_buf = torch.empty_like(q_ring[0])
    q_buf.copy_(q_ring[0])
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(echo.NUM_STAGES + 1)]
    for e in evs:
        e.record()
    mk = lambda events=None: echo.make_step_args(pool, ws, q_buf, w, k_index, ctx, r2h, K_TOP, out, stage=stage,
                                                s_hat=s_hat if stage is not None else None, clock_dev=clock,
                                                advance_clock=True, stats=stats, events=events)
    a_step, a_stage = mk(), mk(evs)
    echo.echo_decode_step(a_step)
    torch.cuda.synchronize()
    g_step = capture_graph(torch, lambda: echo.echo_decode_step(a_step))
    g_stage = capture_graph(torch, lambda: echo.echo_decode_step(a_stage))
    replay_timed(torch, g_step, lambda i: q_buf.copy_(q_ring[1 + i]), flush_l2, warmup - 1)
    stats.t.zero_()
    out.dev_status.zero_()
    ms = replay_timed(torch, g_step, lambda i: q_buf.copy_(q_ring[warmup + i]), flush_l2, n_timed)
    sv = stats.as_dict()
    status = int(out.dev_status.item())
    per = {name: [] for name in ("append", "indexer", "topk", "recall", "ema")}
    for i in range(n_stage):
        q_buf.copy_(q_ring[warmup + n_timed + i])
        flush_l2()
        g_stage.replay()
        torch.cuda.synchronize()
        for j, name in enumerate(per):
            per[name].append(evs[j].elapsed_time(evs[j + 1]))
    stage_ms = {name: float(np.mean(v)) for name, v in per.items()}
    idx_bytes = B_ * L_ * (128 + 4) + B_ * (64 * 128 + 64 * 4)
    rec_rows = sv["recalled"] / n_timed
    rec_gbs = rec_rows * 1152 / (stage_ms["recall"] * 1e-3) / 1e9
    res = {"B": B_, "L": L_, "overlap": overlap, "rho": rho, "mode": mode, "steps": n_timed,
           "value": 1e3 / float(np.mean(ms)), "unit": "steps/s", "ms_per_step": float(np.mean(ms)),
           "step_us_p50": float(np.median(ms)) * 1e3, "step_us_p90": float(np.percentile(ms, 90)) * 1e3,
           "step_us_max": float(np.max(ms)) * 1e3, "scored_tokens_per_s": B_ * L_ * 1e3 / float(np.mean(ms)),
           "hit_rate": sv["hits"] / max(1, sv["unique_rows"]), "recalled_rows_per_step": rec_rows,
           "prefetched_rows_per_step": sv["staged"] / n_timed, "stage_ms": stage_ms,
           "indexer": {"bytes": idx_bytes, "gbs": idx_bytes / (stage_ms["indexer"] * 1e-3) / 1e9,
                       "frac": idx_bytes / (stage_ms["indexer"] * 1e-3) / 1e9 / hbm_peak},
           "recall": {"bytes_per_step": rec_rows * 1152, "gbs": rec_gbs, "frac_h2d": rec_gbs / h2d_gbs,
                      "source": "host pool" if mode == "off" else "host pool and prefetched rows"},
           "dev_status": status}
    del k_index, q_ring, pool, ws, stage, out
    return res


# (B, L, consecutive top-k overlap): overlap 0.7 gives a hit rate near 0.9 at recall (rows
# selected a few steps back are often still resident); the last two are the large-volume
# recall points (B >= 16, hit rate <= 0.7)
SWEEP_POINTS = [(1, 16384, 0.7), (1, 131072, 0.7), (8, 16384, 0.7), (8, 131072, 0.7), (32, 16384, 0.7),
                (32, 131072, 0.7), (16, 65536, 0.5), (32, 131072, 0.5)]


def multistep_leg(echo, torch, flush_l2, host_big, n_steps=256, layers=4, B_=16, L0=32768, n_g=100_000,
                  overlap=0.85, seed=500):
    """The multi-step configuration: `layers` layers' decode steps with write-through appends in
    ONE captured graph, replayed for n_steps consecutive steps (context L0 -> L0 + n_steps),
    a full 100K-slot pool per layer, step-correlated queries.  Inputs of each step (queries, new
    tokens) are copied into the graph's buffers outside the events; L2 is flushed between
    steps."""
    rho = rho_for(L0, overlap)
    L_max = L0 + n_steps
    n_h = B_ * L_max
    lay = []
    for l in range(layers):
        k_index, qf, w, g = gpu_indexer_inputs(torch, B_, 1, L_max, seed + l)
        st = None
        from sparse_attention_kv_fp8_gb300 import workload as wl
        idx = np.sort(np.random.default_rng(seed + l).choice(B_ * L0, size=n_g, replace=False))
        rows = (idx // L0) * L_max + idx % L0
        st = wl.resident_pool(n_g, n_h, rows, wl.random_clocks(n_g, T0, seed + l), seed + l)
        pool = echo.Pool(n_g, host_big[l * n_h:(l + 1) * n_h])
        pool.load_state(st, gpu_kv=pool.gpu_kv)
        d = dict(k=k_index, w=w, pool=pool, ws=echo.Workspace(n_g, B_ * K_TOP),
                 stage=echo.Stage(B_, (L_max + CAP_DIV - 1) // CAP_DIV, CAP_DIV, while_scoring=True),
                 out=echo.StepBuffers(B_, 1, L_max, K_TOP), stats=echo.Stats(),
                 s_hat=torch.full((B_, 1), float("inf"), dtype=torch.float32, device="cuda"),
                 clock=torch.tensor([T0], dtype=torch.int32, device="cuda"),
                 ctx=torch.full((B_,), L0, dtype=torch.int32, device="cuda"),
                 q_ring=gpu_query_ring(torch, qf, rho, n_steps, g),
                 kv_ring=(torch.randn((n_steps, B_, 576), generator=g, device="cuda").to(torch.bfloat16)
                          .view(torch.int16)),
                 ki_ring=(torch.randn((n_steps, B_, 128), generator=g, device="cuda").clamp_(-8, 8)
                          .to(torch.float8_e4m3fn).view(torch.uint8)))
        d["q_buf"] = torch.empty_like(d["q_ring"][0])
        d["kv_buf"] = torch.empty_like(d["kv_ring"][0])
        d["ki_buf"] = torch.empty_like(d["ki_ring"][0])
        d["r2h"] = torch.arange(n_h, dtype=torch.int32, device="cuda").view(B_, L_max)
        d["args"] = echo.make_step_args(d["pool"], d["ws"], d["q_buf"], w, k_index, d["ctx"], d["r2h"], K_TOP,
                                        d["out"], stage=d["stage"], s_hat=d["s_hat"], new_kv=d["kv_buf"],
                                        new_k_index=d["ki_buf"], clock_dev=d["clock"], advance_clock=True,
                                        stats=d["stats"])
        lay.append(d)

    def set_inputs(t):
        for d in lay:
            d["q_buf"].copy_(d["q_ring"][t])
            d["kv_buf"].copy_(d["kv_ring"][t])
            d["ki_buf"].copy_(d["ki_ring"][t])

    def run_all():
        for d in lay:
            echo.echo_decode_step(d["args"])

    set_inputs(0)
    run_all()          # step 0 eagerly (kernel attributes), then one graph of all layers
    torch.cuda.synchronize()
    g_all = capture_graph(torch, run_all)
    for d in lay:
        d["stats"].t.zero_()
        d["out"].dev_status.zero_()
    ms = replay_timed(torch, g_all, lambda i: set_inputs(1 + i), flush_l2, n_steps - 1)
    sv = [d["stats"].as_dict() for d in lay]
    status = 0
    for d in lay:
        status |= int(d["out"].dev_status.item())
    ctx_end = int(lay[0]["ctx"][0].item())
    kbytes = layers * B_ * (L0 + n_steps / 2) * 128
    res = {"layers": layers, "B": B_, "L": f"{L0} -> {ctx_end}", "overlap": overlap, "rho": rho,
           "steps": len(ms), "graph": f"one CUDA graph of {layers} layers' decode steps with appends",
           "value": 1e3 / float(np.mean(ms)), "unit": "steps/s (all layers)", "ms_per_step": float(np.mean(ms)),
           "ms_per_layer_step": float(np.mean(ms)) / layers, "step_us_p50": float(np.median(ms)) * 1e3,
           "kI_gbs": kbytes / (float(np.mean(ms)) * 1e-3) / 1e9,
           "hit_rate": sum(x["hits"] for x in sv) / max(1, sum(x["unique_rows"] for x in sv)),
           "recalled_rows_per_layer_step": sum(x["recalled"] for x in sv) / (layers * len(ms)),
           "appended_per_layer_step": sum(x["appended"] for x in sv) / (layers * len(ms)),
           "dev_status": status}
    del lay
    return res


def mtp_leg(echo, torch, flush_l2, host_big, hbm_peak, h2d_gbs, n_timed=12, warmup=3, B_=32, n_q=2, L_=100_000,
            n_g=65536, sub=8, overlap=0.5, seed=71):
    """The HBM-pressure / MTP configuration: B_ = 32 requests, two query tokens each, context
    100000, a 65536-slot pool, 3.2M host rows.  One step = indexer (no prefetch) -> top-k of the
    64 rows -> the recall in four sub-batches of 8 requests (each at its own clock: its rows are
    protected while it is recalled, evictable for the next), all in one graph with stage events.
    Indexer bytes: B_ L_ 128 + B_ n_q L_ 4 + q / w; recall: 1152 per recalled row from the host."""
    rho = rho_for(L_, overlap)
    k_index, qf, w, g = gpu_indexer_inputs(torch, B_, n_q, L_, seed)
    q_ring = gpu_query_ring(torch, qf, rho, warmup + n_timed + 1, g)
    n_h = B_ * L_
    r2h = torch.arange(n_h, dtype=torch.int32, device="cuda").view(B_, L_)
    ctx = torch.full((B_,), L_, dtype=torch.int32, device="cuda")
    pool = echo.Pool(n_g, host_big[:n_h])
    pool.load_state(pool_state_for(n_g, n_h, seed), gpu_kv=pool.gpu_kv)
    nsub = B_ // sub
    ws = echo.Workspace(n_g, sub * n_q * K_TOP)
    scores = torch.empty((B_, n_q, L_), dtype=torch.float32, device="cuda")
    sel = torch.empty((B_, n_q, K_TOP), dtype=torch.int32, device="cuda")
    kth = torch.empty((B_, n_q), dtype=torch.float32, device="cuda")
    out = torch.empty_like(sel)
    stats = echo.Stats()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    clocks = torch.zeros(nsub, dtype=torch.int32, device="cuda")
    q_buf = torch.empty_like(q_ring[0])
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nsub + 3)]
    for e in evs:
        e.record()

    def step(events):
        if events:
            evs[0].record()
        echo.echo_indexer_score(q_buf, w, k_index, ctx, scores, dev_status=status)
        if events:
            evs[1].record()
        echo.echo_select_topk(scores, ctx, K_TOP, sel, kth)
        if events:
            evs[2].record()
        for s_ in range(nsub):
            bs = slice(s_ * sub, (s_ + 1) * sub)
            echo.echo_prefetch_recall(pool, ws, sel[bs], r2h[bs], ctx[bs], 0, out[bs], stats=stats, dev_status=status,
                                      clock_dev=clocks[s_:s_ + 1])
            if events:
                evs[3 + s_].record()

    def before(t):
        q_buf.copy_(q_ring[t])
        clocks.copy_(torch.arange(nsub, dtype=torch.int32, device="cuda") + (T0 + nsub * t))

    before(0)
    step(False)
    torch.cuda.synchronize()
    g_step = capture_graph(torch, lambda: step(False))
    replay_timed(torch, g_step, lambda i: before(1 + i), flush_l2, warmup - 1)
    stats.t.zero_()
    ms = replay_timed(torch, g_step, lambda i: before(warmup + i), flush_l2, n_timed)
    sv = stats.as_dict()
    # stage times: one more step launched directly with events between the calls (indexer,
    # top-k, recall sub-batches; the launches queue ahead of the GPU)
    before(warmup + n_timed)
    flush_l2()
    st0 = stats.as_dict()
    torch.cuda._sleep(2_000_000)
    step(True)
    torch.cuda.synchronize()
    st1 = stats.as_dict()
    idx_ms = evs[0].elapsed_time(evs[1])
    topk_ms = evs[1].elapsed_time(evs[2])
    rec_ms = evs[2].elapsed_time(evs[2 + nsub])
    idx_bytes = B_ * L_ * 128 + B_ * n_q * L_ * 4 + B_ * n_q * (64 * 128 + 64 * 4)
    rec_rows = st1["recalled"] - st0["recalled"]
    rec_gbs = rec_rows * 1152 / (rec_ms * 1e-3) / 1e9
    res = {"B": B_, "n_q": n_q, "L": L_, "n_g": n_g, "n_h": n_h, "overlap": overlap, "rho": rho,
           "recall_sub_batches": nsub, "steps": n_timed, "value": 1e3 / float(np.mean(ms)), "unit": "steps/s",
           "ms_per_step": float(np.mean(ms)), "scored_tokens_per_s": B_ * n_q * L_ * 1e3 / float(np.mean(ms)),
           "hit_rate": sv["hits"] / max(1, sv["unique_rows"]), "recalled_rows_per_step": sv["recalled"] / n_timed,
           "evicted_per_step": sv["evicted"] / n_timed,
           "stage_ms": {"indexer": idx_ms, "topk": topk_ms, "recall": rec_ms},
           "indexer": {"bytes": idx_bytes, "gbs": idx_bytes / (idx_ms * 1e-3) / 1e9,
                       "frac": idx_bytes / (idx_ms * 1e-3) / 1e9 / hbm_peak},
           "recall": {"rows": rec_rows, "bytes": rec_rows * 1152, "gbs": rec_gbs, "frac_h2d": rec_gbs / h2d_gbs,
                      "source": "host pool (prefetch off)"},
           "dev_status": int(status.item())}
    del k_index, scores, pool, ws
    return res


def warm_host_translations(echo, torch, host_t, page_bytes=0):
    """Read the pinned host pool through the recall kernel before timing -- every row by
    default, else one row per `page_bytes` -- so the GPU has translated every page and
    the pool's lines have made one trip over the host link since the CPU wrote them (in
    serving the pool is read every step; a cold translation costs far more than the
    read, and on freshly written pages the first reads were seen to run several times
    slower for about a second)."""
    n_h = host_t.shape[0]
    step = max(1, page_bytes // (host_t.shape[1] * 2))
    rows = np.arange(0, n_h, step, dtype=np.int32)
    pool = echo.Pool(rows.size, host_t)
    echo.echo_pool_init(pool)
    ws = echo.Workspace(rows.size, rows.size)
    r2h = torch.from_numpy(rows.reshape(1, -1)).cuda()
    sel = torch.arange(rows.size, dtype=torch.int32, device="cuda").view(1, 1, -1)
    ctx = torch.tensor([rows.size], dtype=torch.int32, device="cuda")
    out = torch.empty_like(sel)
    echo.echo_prefetch_recall(pool, ws, sel, r2h, ctx, 1, out)
    torch.cuda.synchronize()


def recall_bandwidth_probe(echo, torch, host_t, flush_l2, rows=65536, n_g=65536):
    """Recall of `rows` distinct non-resident host rows into an empty pool, prefetch
    off: host-link bytes over the copy time (the recall call's three kernels)."""
    pool = echo.Pool(n_g, host_t)
    echo.echo_pool_init(pool)
    ws = echo.Workspace(n_g, rows)
    g = np.random.default_rng(5)
    pick = np.sort(g.choice(B * L, size=rows, replace=False)).astype(np.int32)
    r2h = torch.from_numpy(pick.reshape(1, rows)).cuda()
    sel = torch.arange(rows, dtype=torch.int32, device="cuda").view(1, 1, rows)
    ctx = torch.tensor([rows], dtype=torch.int32, device="cuda")
    out = torch.empty_like(sel)
    best = 1e9
    for it in range(4):
        echo.echo_pool_init(pool)
        flush_l2()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        echo.echo_prefetch_recall(pool, ws, sel, r2h, ctx, 10 + it, out)
        a1.record()
        torch.cuda.synchronize()
        best = min(best, a0.elapsed_time(a1))
    ok = bool((out >= 0).all().item())
    return {"rows": rows, "bytes": rows * 1152, "ms": best, "gbs": rows * 1152 / (best * 1e-3) / 1e9, "all_recalled": ok}


def block_recall_probe(echo, torch, flush_l2, h2d_gbs, B_req=4, n_blocks=1024, n_g=8192, reps=4):
    """The block-level / GQA variant of the cache manager: a pool row is one block of 64
    tokens of one KV head (K and V, 128 dims: 32 KB), a selection row one (request, KV
    head) pair: 4 requests x 8 KV heads, 1024 blocks each (64K tokens).
    cold: 64 blocks per selection row (2048 rows, 64 MiB) recalled into an empty pool,
      all misses: host-link bytes over the call's time, best of `reps`.
    steady: the pool full of older blocks at the start (every miss evicts); NSA-style 16
      blocks per row, block scores of consecutive steps correlated (rho 0.9); GPU top-k
      plus recall per step, median over the steps after the first 4."""
    from sparse_attention_kv_fp8_gb300 import workload as wl
    R = wl.block_row_elems()
    rows = B_req * wl.GQA_KV_HEADS
    n_h = rows * n_blocks
    host = torch.empty((n_h, R), dtype=torch.int16, pin_memory=True)
    host[:, :8] = torch.arange(n_h, dtype=torch.int32).view(-1, 1).to(torch.int16)   # rows told apart
    host[:, 8:] = 1
    pool = echo.Pool(n_g, host)
    echo.echo_pool_init(pool)
    ws = echo.Workspace(n_g, rows * 64)
    r2h = torch.from_numpy(wl.req_to_host(rows, n_blocks)).cuda()
    ctx = torch.full((rows,), n_blocks, dtype=torch.int32, device="cuda")
    g = np.random.default_rng(6)
    sel = torch.from_numpy(np.sort(np.stack([g.choice(n_blocks, 64, replace=False) for _ in range(rows)]), axis=1)
                           .astype(np.int32)[:, None, :]).cuda()
    out = torch.empty_like(sel)
    best = 1e9
    for it in range(reps):
        echo.echo_pool_init(pool)
        flush_l2()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        echo.echo_prefetch_recall(pool, ws, sel, r2h, ctx, 10 + it, out)
        a1.record()
        torch.cuda.synchronize()
        best = min(best, a0.elapsed_time(a1))
    cold_ok = bool((out >= 0).all().item())
    cold_bytes = rows * 64 * R * 2
    # steady decode steps at block granularity, from a full pool
    res = wl.random_resident_rows(n_h, n_g, 6)
    pool.load_state(wl.resident_pool(n_g, n_h, res, wl.random_clocks(n_g, 100, 6), 6))
    k = wl.GQA_TOPK_BLOCKS
    scores = [torch.from_numpy(sc).cuda() for sc in wl.block_scores(rows, n_blocks, 7, 12, 0.9)]
    sel_k = torch.empty((rows, 1, k), dtype=torch.int32, device="cuda")
    kth = torch.empty((rows, 1), dtype=torch.float32, device="cuda")
    out_k = torch.empty_like(sel_k)
    stats = echo.Stats()
    ts, before = [], None
    for t, sc in enumerate(scores):
        if t == 4:
            torch.cuda.synchronize()
            before = stats.as_dict()
        flush_l2()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        echo.echo_select_topk(sc, ctx, k, sel_k, kth)
        echo.echo_prefetch_recall(pool, ws, sel_k, r2h, ctx, 100 + t, out_k, stats=stats)
        a1.record()
        torch.cuda.synchronize()
        if t >= 4:
            ts.append(a0.elapsed_time(a1))
    after = stats.as_dict()
    uniq = max(1, after["unique_rows"] - before["unique_rows"])
    return {"row_bytes": R * 2, "selection_rows": rows, "blocks_per_row": n_blocks,
            "cold": {"rows": rows * 64, "bytes": cold_bytes, "ms": best, "gbs": cold_bytes / (best * 1e-3) / 1e9,
                     "frac_h2d": cold_bytes / (best * 1e-3) / 1e9 / h2d_gbs, "all_recalled": cold_ok},
            "steady": {"k_blocks": k, "us_per_step": float(np.median(ts)) * 1e3,
                       "hit_rate": (after["hits"] - before["hits"]) / uniq,
                       "recalled_rows_per_step": (after["recalled"] - before["recalled"]) / len(ts)}}


def indexer_volume_probe(echo, torch, inp, flush_l2, hbm_peak, batches=(8, 24, 64), reps=5):
    """The indexer alone (scoring, no prefetch) at growing per-launch volume: the decode
    batch's keys tiled to B requests, L2 flushed before each launch, median of `reps`
    CUDA-event timings.  Shows the fixed launch cost giving way to bandwidth."""
    res = []
    B0, L_ = inp.k_index.shape[0], inp.k_index.shape[1]
    for Bv in batches:
        idx = np.arange(Bv) % B0
        k_t = torch.from_numpy(np.ascontiguousarray(inp.k_index[idx])).cuda()
        q_t = torch.from_numpy(np.ascontiguousarray(inp.q[idx])).cuda()
        w_t = torch.from_numpy(np.ascontiguousarray(inp.w[idx])).cuda()
        ctx_t = torch.full((Bv,), L_, dtype=torch.int32, device="cuda")
        sc = torch.empty((Bv, 1, L_), dtype=torch.float32, device="cuda")
        echo.echo_indexer_score(q_t, w_t, k_t, ctx_t, sc)
        ts = []
        for _ in range(reps):
            flush_l2()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            echo.echo_indexer_score(q_t, w_t, k_t, ctx_t, sc)
            a1.record()
            torch.cuda.synchronize()
            ts.append(a0.elapsed_time(a1))
        ms = float(np.median(ts))
        nbytes = Bv * L_ * 128 + Bv * L_ * 4 + Bv * (64 * 128 + 64 * 4)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res.append({"B": Bv, "L": L_, "bytes": nbytes, "us": ms * 1e3, "gbs": gbs, "frac": gbs / hbm_peak})
        del k_t, sc
    return res


def prefill_probe(echo, torch, flush_l2, B=1, L_=32768, C=512, k=K_TOP, reps=3, seed=21):
    """The prefill chunk indexer (the last C tokens of each request as queries, causal):
    scores only, then with the approximate top-k (shift = the k-th score of the chunk's
    last query).  Median CUDA-event time of `reps` launches, L2 flushed before each.
    FLOP = 2 * 64 * 128 per (query, visible key)."""
    from sparse_attention_kv_fp8_gb300 import workload as wl
    inp = wl.indexer_inputs(B, C, L_, L_, seed=seed)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q, w, k_index, ctx = dev(inp.q), dev(inp.w), dev(inp.k_index), dev(inp.ctx_len)
    scores = torch.empty((B, C, L_), dtype=torch.float32, device="cuda")
    thr = torch.empty((B, C), dtype=torch.int32, device="cuda")
    sub = torch.empty((B, C), dtype=torch.int32, device="cuda")
    echo.echo_prefill_indexer_score(q, w, k_index, ctx, scores)
    torch.cuda.synchronize()
    last = scores[:, C - 1, :].cpu().numpy()
    shift = torch.from_numpy(np.array([np.sort(last[b])[::-1][k - 1] for b in range(B)], np.float32)).cuda()

    def timed(fn):
        ts = []
        for _ in range(reps):
            flush_l2()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            fn()
            a1.record()
            torch.cuda.synchronize()
            ts.append(a0.elapsed_time(a1))
        return float(np.median(ts))

    def busy():
        flush_l2()
        torch.cuda.synchronize()

    with ClockSampler(torch.cuda.current_device(), busy=busy) as clk:
        t0 = time.time()
        ms_plain = timed(lambda: echo.echo_prefill_indexer_score(q, w, k_index, ctx, scores))
        ms_approx = timed(lambda: echo.echo_prefill_indexer_score(q, w, k_index, ctx, scores, s_shift=shift, k=k,
                                                                  thr_bin=thr, subset_n=sub))
        clk.window(t0, time.time())
    pairs = int(sum(max(0, int(inp.ctx_len[b]) - (C - 1 - i)) for b in range(B) for i in range(C)))
    flop = 2.0 * 64 * 128 * pairs
    return {"B": B, "L": L_, "C": C, "k": k, "query_key_pairs": pairs, "flop": flop,
            "ms_scores": ms_plain, "tflops_scores": flop / (ms_plain * 1e-3) / 1e12,
            "ms_with_approx_topk": ms_approx, "tflops_with_approx_topk": flop / (ms_approx * 1e-3) / 1e12,
            "mean_subset_of_k": float(sub.float().mean().item()) / k, "clocks": clk.summary()}


def mla_probe(echo, torch, flush_l2, pool, out_slot, hbm_peak, bf16_peak, reps=5, seed=31):
    """Sparse MLA decode over the decode step's own selection (out_slot of the last
    timed step, rows in the step's GPU pool): 128 heads x 576-dim absorbed queries.
    Median CUDA-event time of `reps` graph replays (both kernels), L2 flushed before each.
    FLOP = 2 * 128 * (576 + 512) per (query token, selected row); algorithmic bytes =
    the selected rows (1152 B each) + q + out + lse."""
    from sparse_attention_kv_fp8_gb300 import workload as wl
    Bq, n_q, k = out_slot.shape
    q = torch.from_numpy(wl.mla_queries(Bq, n_q, seed).view(np.int16)).cuda()
    out = torch.empty((Bq, n_q, 128, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((Bq, n_q, 128), dtype=torch.float32, device="cuda")
    ws = echo.MlaWorkspace(Bq, n_q, k)
    scale = 1.0 / float(np.sqrt(192.0))
    echo.echo_sparse_mla_decode(q, pool.gpu_kv, out_slot, scale, out, lse, ws)
    torch.cuda.synchronize()
    # replayed from a CUDA graph, as inside a captured decode step (no host launch work
    # between the events)
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g, stream=cap):
            echo.echo_sparse_mla_decode(q, pool.gpu_kv, out_slot, scale, out, lse, ws)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush_l2()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        g.replay()
        a1.record()
        torch.cuda.synchronize()
        ts.append(a0.elapsed_time(a1))
    ms = float(np.median(ts))
    rows = int((out_slot >= 0).sum().item())
    flop = 2.0 * 128 * (576 + 512) * rows
    nbytes = rows * 1152 + q.numel() * 2 + out.numel() * 4 + lse.numel() * 4
    return {"B": Bq, "n_q": n_q, "k": k, "rows": rows, "us": ms * 1e3,
            "tflops": flop / (ms * 1e-3) / 1e12, "frac_bf16_peak": flop / (ms * 1e-3) / 1e12 / bf16_peak,
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm_peak,
            "workspace_bytes": ws.bytes}


def run_kernel_case(args):
    """Single-kernel case for profilers: the indexer with the fused prefetch
    (threshold = each row's k-th score, 97% of the top-k resident) on B x L tokens,
    `--reps` launches after one without prefetch."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import sparse_attention_kv_fp8_gb300 as echo
    from sparse_attention_kv_fp8_gb300 import workload as wl
    Bk, Lk = args.B, args.L
    if args.kernel == "mla":
        # the decode shape's selection over a full 200K-slot pool of random rows
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        pool_kv = torch.from_numpy(wl.bf16_encode(np.random.default_rng(7).standard_normal(
            (N_G, echo.KV_ELEMS), dtype=np.float32)).view(np.int16)).cuda()

        class _Pool:
            gpu_kv = pool_kv
        g = np.random.default_rng(8)
        sl = torch.from_numpy(np.stack([g.choice(N_G, size=args.k, replace=False) for _ in range(Bk)])
                              .astype(np.int32)[:, None, :]).cuda()
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        res = mla_probe(echo, torch, flush.zero_, _Pool, sl, float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"]),
                        reps=args.reps)
        print(json.dumps({"kernel_case": "mla", **res}))
        return 0
    if args.kernel == "prefill":
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        res = prefill_probe(echo, torch, flush.zero_, B=Bk, L_=Lk, C=args.C, reps=args.reps)
        print(json.dumps({"kernel_case": "prefill", **res}))
        return 0
    inp = wl.indexer_inputs(Bk, 1, Lk, Lk, seed=3)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n_h = Bk * Lk
    host_t = torch.zeros((n_h, echo.KV_ELEMS), dtype=torch.int16, pin_memory=True)
    pool = echo.Pool(min(n_h, 200_000), host_t)
    echo.echo_pool_init(pool)
    stage = echo.Stage(Bk, Lk // CAP_DIV, CAP_DIV)
    q, w, k_index, ctx, r2h = dev(inp.q), dev(inp.w), dev(inp.k_index), dev(inp.ctx_len), dev(wl.req_to_host(Bk, Lk))
    scores = torch.empty((Bk, 1, Lk), dtype=torch.float32, device="cuda")
    sel = torch.empty((Bk, 1, K_TOP), dtype=torch.int32, device="cuda")
    kth = torch.empty((Bk, 1), dtype=torch.float32, device="cuda")
    echo.echo_indexer_score(q, w, k_index, ctx, scores)
    echo.echo_select_topk(scores, ctx, K_TOP, sel, kth)
    # make 97% of each row's top-k resident (the decode workload's hit rate), so the
    # fused prefetch moves about as many rows per tile as in the benchmark
    sel_np = sel.cpu().numpy()
    g = np.random.default_rng(4)
    rows = [int(b * Lk + p) for b in range(Bk) for p in sel_np[b, 0] if p >= 0 and g.random() < 0.97]
    rows = rows[:pool.n_g]
    ws = echo.Workspace(pool.n_g, len(rows))
    out = torch.empty(len(rows), dtype=torch.int32, device="cuda")
    warm_host_translations(echo, torch, host_t)
    echo.echo_pool_alloc(pool, ws, torch.tensor(rows, dtype=torch.int32, device="cuda"),
                         torch.tensor([len(rows)], dtype=torch.int32, device="cuda"), 1, out)
    for _ in range(args.reps):
        stage.count.zero_()
        echo.echo_indexer_score(q, w, k_index, ctx, scores, s_hat=kth, req_to_host=r2h, pool=pool, stage=stage)
    torch.cuda.synchronize()
    print(json.dumps({"kernel_case": "indexer", "B": Bk, "L": Lk, "reps": args.reps,
                      "staged": int(stage.count.clamp(max=Lk // CAP_DIV).sum().item())}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-requests", type=int, default=B)
    ap.add_argument("--e2e-steps", type=int, default=200, help="steps of the wall-clock e2e measurement")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other configurations (sweep, multi-step, HBM-pressure / MTP, overlap 0.7)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overlap", type=float, default=TARGET_OVERLAP,
                    help="consecutive top-k overlap of the synthetic queries (0.5, 0.7, 0.9 or 0.99)")
    ap.add_argument("--reserve", type=int, default=8192,
                    help="slots per recall for the direct-to-slot comparison leg (0: skip it and the "
                         "no-prefetch leg)")
    ap.add_argument("--prefetch-tail", action="store_true",
                    help="let the prefetch also copy candidates still queued when scoring ends (default: "
                         "dropped, the recall fetches them if selected)")
    ap.add_argument("--kernel", default=None, choices=[None, "indexer", "prefill", "mla"],
                    help="run one kernel on a small case (for profilers) instead of the benchmark")
    ap.add_argument("--B", type=int, default=24)
    ap.add_argument("--L", type=int, default=65536)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--C", type=int, default=512, help="queries per request of the prefill kernel case")
    ap.add_argument("--k", type=int, default=K_TOP, help="selected rows per query of the MLA kernel case")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.kernel:
        return run_kernel_case(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
