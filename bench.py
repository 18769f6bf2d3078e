"""Benchmark of the rational-softmax attention hot path on GB300.

One step = the whole hot path over one batch of seeded synthetic input:
  ra_softmax      fp32 logits [16384, 8192] ~ N(0, 4^2)
  ra_attention    forward + backward, B=4, H=16, N=8192, D=128, bf16, Q,K ~ N(0, 3^2),
                  V, dO ~ N(0, 1), scale 1/sqrt(128), non-causal (fp32 outputs/gradients)
value = counted attention FLOPs of the step / step time (standard-attention count:
forward 4 B H N^2 D, backward 2.5x forward), in TFLOP/s.  ra_softmax's GB/s, the
per-call times and a causal long-sequence forward (B=4, H=16, N=8192, D=128) are
reported beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the float64 CPU oracle (the only reference that exists
for this method) on a bounded sample of the same workload.  Under torchrun each
rank runs the full step on its own GPU (weak scaling; the path has no exchange).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ra_attention fwd/bwd TFLOP/s and % bf16 TC peak; ra_softmax GB/s vs HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def attn_flops(B, H, NQ, NK, D, causal, backward):
    f = 4.0 * B * H * NQ * NK * D * (0.5 if causal else 1.0)
    return f * (3.5 if backward else 1.0)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(value, dist, device):
    """The largest value over all ranks (the slowest rank's time); the value itself on one rank."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world, flops_per_rank_step, steps, elapsed_ms):
    """TFLOP/s of the whole job: every rank runs the same step (weak scaling), and the
    elapsed time is the slowest rank's."""
    return world * flops_per_rank_step * steps / (elapsed_ms * 1e-3) / 1e12


def step_config(w, sw):
    """The workload of one step (both arms report the same)."""
    return {
        "workload": "ra_softmax fp32 [16384, 8192] sigma 4 + ra_attention fwd+bwd B4 H16 N8192 D128 bf16 "
                    "Q,K sigma 3 scale 1/sqrt(128) non-causal (fp32 O and gradients)",
        "ra_softmax": {"rows": sw.rows, "cols": sw.cols, "sigma": sw.sigma, "dtype": "f32"},
        "attention": {"B": w.B, "H": w.H, "N": w.N, "D": w.D, "sigma_qk": w.sigma_qk, "causal": w.causal,
                      "dtype": "bf16 in, fp32 accumulate, fp32 out"},
        "l2": "no flush: each step reads > 1.5 GiB of inputs, above the 129 MB L2",
        "per_gpu": "each rank runs the whole step on its own GPU (no exchange on this path)",
    }


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def _ptr(t):
    import ctypes
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class HotPath:
    """Preallocated device buffers and the C-ABI calls of one step.

    Inputs and outputs come in two device sets, so that the end-to-end loop can copy the
    next step's inputs in (and the last step's results out) while a step computes.  The
    row statistics and workspaces are used only inside a step, on the compute stream, and
    exist once."""

    def __init__(self, dev, host_inputs, w, sw):
        import ctypes

        import torch

        import rational_softmax_attention_gb300 as ra
        self.torch, self.ra, self.ctypes = torch, ra, ctypes
        self.L = ra.lib()
        self.dev = dev
        self.w, self.sw = w, sw
        self.host_in = host_inputs
        B, H, N, D = host_inputs[0].shape
        f32 = torch.float32
        self.sets = []
        for _ in range(2):
            dev_in = [t.to(dev) for t in host_inputs]
            o = torch.empty((B, H, N, D), dtype=f32, device=dev)
            dq = torch.empty((B, H, N, D), dtype=f32, device=dev)
            outs = [o, dq, torch.empty_like(dq), torch.empty_like(dq), torch.empty_like(dev_in[4])]
            self.sets.append((dev_in, outs))
        self.dev_in, self.outs = self.sets[0]
        self.rm = torch.empty((B, H, N), dtype=f32, device=dev)
        self.rs = torch.empty((B, H, N), dtype=f32, device=dev)
        self.ra_ = torch.empty((B, H, N), dtype=torch.int32, device=dev)
        self.ws = torch.empty(self.L.ra_attention_bwd_workspace_size(B, H, N, N, D), dtype=torch.uint8, device=dev)
        self.fws = torch.empty(self.L.ra_attention_fwd_workspace_size(B, H, N, N, D), dtype=torch.uint8, device=dev)
        self.host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in self.outs]
        self.shape = (B, H, N, D)

    def _check(self, name, code):
        if code != 0:
            raise RuntimeError(f"{name}: {self.L.ra_status_string(code).decode()}")

    def softmax(self, st, b=0):
        x = self.sets[b][0][4]
        y = self.sets[b][1][4]
        self._check("ra_softmax_fwd", self.L.ra_softmax_fwd(_ptr(x), _ptr(y), x.shape[0], x.shape[1], 0, st))

    def fwd(self, st, counts=None, b=0):
        q, k, v, _, _ = self.sets[b][0]
        o = self.sets[b][1][0]
        B, H, N, D = self.shape
        self._check("ra_attention_fwd", self.L.ra_attention_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(self.rm), _ptr(self.rs), _ptr(self.ra_), _ptr(counts),
            _ptr(self.fws), B, H, N, N, D, float(self.w.scale), int(self.w.causal), 1, 0, st))

    def bwd(self, st, b=0):
        q, k, v, do, _ = self.sets[b][0]
        o, dq, dk, dv, _ = self.sets[b][1]
        B, H, N, D = self.shape
        self._check("ra_attention_bwd", self.L.ra_attention_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(self.rm), _ptr(self.rs), _ptr(self.ra_),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(self.ws), B, H, N, N, D, float(self.w.scale),
            int(self.w.causal), 1, 0, 0, st))

    def step(self, st, events=None, b=0):
        """One step.  events (optional): {"sm": e, "fwd": [3 events], "bwd": [4 events]}; the
        library records the call's events at its kernel boundaries (ra_debug_kernel_events)."""
        if events:
            events["sm"].record()
        self.softmax(st, b)
        if events:
            self.ra.debug_kernel_events(events["fwd"])
        self.fwd(st, None, b)
        if events:
            self.ra.debug_kernel_events(events["bwd"])
        self.bwd(st, b)
        if events:
            self.ra.debug_kernel_events(None)

    def run_e2e(self, stream, steps):
        """`steps` end-to-end steps, timed with events on `stream`, returned in ms.

        Step i copies its inputs from pinned host memory into device set i % 2 on an H2D
        stream, computes on `stream`, and copies every output back to pinned host memory
        on a D2H stream.  Set b is refilled only after the step that last read it has
        finished, and recomputed only after its previous results have left the device.
        The closing event waits for the last D2H copy, so every step's copies lie inside
        the timed region."""
        torch = self.torch
        st = self.ctypes.c_void_p(stream.cuda_stream)
        h2d = torch.cuda.Stream(self.dev)
        d2h = torch.cuda.Stream(self.dev)
        done = [torch.cuda.Event() for _ in range(2)]      # step on set b finished
        drained = [torch.cuda.Event() for _ in range(2)]   # outputs of set b copied out
        loaded = [torch.cuda.Event() for _ in range(2)]    # inputs of set b copied in
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d.wait_event(e0)
        d2h.wait_event(e0)
        for i in range(steps):
            b = i % 2
            dev_in, outs = self.sets[b]
            if i >= 2:
                h2d.wait_event(done[b])
            with torch.cuda.stream(h2d):
                for d, h in zip(dev_in, self.host_in):
                    d.copy_(h, non_blocking=True)
            loaded[b].record(h2d)
            stream.wait_event(loaded[b])
            if i >= 2:
                stream.wait_event(drained[b])
            self.step(st, None, b)
            done[b].record(stream)
            d2h.wait_event(done[b])
            with torch.cuda.stream(d2h):
                for h, d in zip(self.host_out, outs):
                    h.copy_(d, non_blocking=True)
            drained[b].record(d2h)
        for b in range(min(2, steps)):
            stream.wait_event(drained[b])
        e1.record(stream)
        torch.cuda.synchronize(self.dev)
        return e0.elapsed_time(e1)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host_in)

    def d2h_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.outs)


def traffic_from_profiles(kernel_tag):
    """DRAM bytes per launch recorded from an ncu capture in profiles/ (None when absent)."""
    path = os.path.join(ROOT, "profiles", "ncu_dram_traffic.txt")
    try:
        with open(path) as fh:
            for ln in fh:
                parts = ln.split()
                if len(parts) >= 2 and parts[0] == kernel_tag:
                    return float(parts[1])
    except OSError:
        pass
    return None


def cpu_oracle_sample(w, sw, q, k, v, do, x, query_rows=8192, softmax_rows=1024, heads=2):
    """Bounded sample of the same workload through the float64 oracle as it stands: the first
    `heads` heads of batch 0, the first `query_rows` queries of each against all keys, forward
    + backward; `softmax_rows` logit rows.  Returns (seconds, counted attention FLOPs,
    description)."""
    import oracle
    xd = x[:softmax_rows].double().numpy()
    dt = 0.0
    for h in range(heads):
        qd = q[0, h, :query_rows].double().numpy()
        dod = do[0, h, :query_rows].double().numpy()
        kd, vd = k[0, h].double().numpy(), v[0, h].double().numpy()
        t0 = time.perf_counter()
        oracle.ra_attention_head_fwd(qd, kd, vd, w.scale, w.causal)
        oracle.ra_attention_head_bwd(qd, kd, vd, dod, w.scale, w.causal)
        dt += time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.ra_softmax(xd)
    dt += time.perf_counter() - t0
    flops = heads * attn_flops(1, 1, query_rows, k.shape[2], k.shape[3], w.causal, True)
    desc = (f"heads (0,0)..(0,{heads - 1}), queries 0..{query_rows - 1} of each against all {k.shape[2]} keys, "
            f"forward+backward in float64, plus ra_softmax of {softmax_rows} logit rows")
    return dt, flops, desc


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = max((i.get("num_threads", 0) for i in threadpool_info()), default=0)
        if n:
            return n
    except Exception:
        pass
    return os.cpu_count()


def run_ours(args):
    import torch

    from rational_softmax_attention_gb300.inputs import (ATTN_LONG_CAUSAL, ATTN_LONG_WIDE, ATTN_MODULE_SHAPE,
                                                         ATTN_TINY_FP32, RA_SOFTMAX_LONG_ROWS, attention_inputs,
                                                         softmax_inputs, workload_inputs)
    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w, sw = ATTN_LONG_WIDE, RA_SOFTMAX_LONG_ROWS
    q, k, v, do = workload_inputs(w)
    x = softmax_inputs(sw.rows, sw.cols, seed=sw.seed, sigma=sw.sigma)
    host_in = [t.pin_memory() for t in (q, k, v, do, x)]
    hp = HotPath(dev, host_in, w, sw)
    stream = torch.cuda.current_stream(dev)
    st = hp.ctypes.c_void_p(stream.cuda_stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # warm-up, then the timed region: exactly `steps` steps, device-resident inputs
    for _ in range(args.warmup):
        hp.step(st)
    barrier()
    def new_ev():
        return torch.cuda.Event(enable_timing=True)
    ev = [{"sm": new_ev(), "fwd": [new_ev() for _ in range(3)], "bwd": [new_ev() for _ in range(4)]}
          for _ in range(args.steps)]
    for e in ev:                      # create every CUDA event before the timed region
        for one in [e["sm"]] + e["fwd"] + e["bwd"]:
            one.record(stream)
    torch.cuda.synchronize(dev)
    t_start, t_end = new_ev(), new_ev()
    with ClockSampler(local) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            hp.step(st, ev[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    status = hp.ra.device_status(stream)
    if status != "RA_OK":
        raise RuntimeError(f"device status after the timed region: {status}")
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    # per call and per kernel, from events on the launching stream (the library records the
    # calls' events between its own launches)
    spans = {
        "ra_softmax_ms": lambda e: e["sm"].elapsed_time(e["fwd"][0]),
        "ra_attention_fwd_ms": lambda e: e["fwd"][0].elapsed_time(e["fwd"][2]),
        "ra_attention_bwd_ms": lambda e: e["bwd"][0].elapsed_time(e["bwd"][3]),
        "bf16_to_f16_kernel (fwd)": lambda e: e["fwd"][0].elapsed_time(e["fwd"][1]),
        "attn_fwd_tc_kernel": lambda e: e["fwd"][1].elapsed_time(e["fwd"][2]),
        "bf16_to_f16_kernel (bwd)": lambda e: e["bwd"][0].elapsed_time(e["bwd"][1]),
        "attn_bwd_dq_tc_kernel": lambda e: e["bwd"][1].elapsed_time(e["bwd"][2]),
        "attn_bwd_dkdv_tc_kernel": lambda e: e["bwd"][2].elapsed_time(e["bwd"][3]),
    }
    med = {kk: statistics.median(fn(e) for e in ev) for kk, fn in spans.items()}
    med["ra_softmax_fwd_vec_kernel"] = med["ra_softmax_ms"]

    B, H, N, D = hp.shape
    flops_step = attn_flops(B, H, N, N, D, w.causal, True)
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_tflops(world, flops_step, args.steps, elapsed_ms)
    fwd_fl = attn_flops(B, H, N, N, D, w.causal, False)
    bwd_fl = flops_step - fwd_fl
    sm_bytes = 2.0 * x.numel() * 4

    # end to end: pinned host inputs -> device, the step, results -> pinned host buffers,
    # with the copies of neighbouring steps overlapping the compute (HotPath.run_e2e)
    hp.run_e2e(stream, max(3, args.warmup))
    barrier()
    e2e_ms = max_over_ranks(hp.run_e2e(stream, args.steps), dist, dev)
    e2e_value = whole_job_tflops(world, flops_step, args.steps, e2e_ms)

    # skipped-tile fraction of the forward (one untimed call with the counters)
    counts = torch.zeros(2, dtype=torch.int64, device=dev)
    hp.fwd(st, counts)
    torch.cuda.synchronize(dev)
    visited, skipped = (int(c) for c in counts.tolist())

    # causal long-sequence forward (reported beside the step; its own timed loop)
    wc = ATTN_LONG_CAUSAL
    qc, kc, vc = (t.to(dev) for t in workload_inputs(wc)[:3])
    oc = torch.empty(qc.shape, dtype=torch.float32, device=dev)
    rmc = torch.empty(qc.shape[:3], dtype=torch.float32, device=dev)
    rsc = torch.empty_like(rmc)
    rac = torch.empty(qc.shape[:3], dtype=torch.int32, device=dev)

    def fwd_causal():
        code = hp.L.ra_attention_fwd(_ptr(qc), _ptr(kc), _ptr(vc), _ptr(oc), _ptr(rmc), _ptr(rsc), _ptr(rac), None,
                                     _ptr(hp.fws), wc.B, wc.H, wc.N, wc.N, wc.D, float(wc.scale), 1, 1, 0, st)
        if code != 0:
            raise RuntimeError("ra_attention_fwd (causal) failed")
    for _ in range(3):
        fwd_causal()
    torch.cuda.synchronize(dev)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(args.steps):
        fwd_causal()
    c1.record(stream)
    torch.cuda.synchronize(dev)
    causal_ms = c0.elapsed_time(c1) / args.steps
    causal_fl = attn_flops(wc.B, wc.H, wc.N, wc.N, wc.D, True, False)
    del qc, kc, vc, oc, rmc, rsc, rac

    # the step's attention with a key-padding mask (the second half of the keys masked for
    # every query): the tile maps leave the padded key tiles out of every kernel
    qm, km, vm, dom = hp.dev_in[:4]
    Bm, Hm, Nm, _ = qm.shape
    kpm = hp.ra.pack_attn_mask((torch.arange(Nm, device=dev) < Nm // 2)[None, :].expand(Nm, Nm), Bm, Hm, Nm, Nm)
    om, rmm, rsm, ram, _ = hp.ra.ra_attention_forward(qm, km, vm, scale=w.scale, out_dtype=torch.float32, mask=kpm)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        return t0.elapsed_time(t1) / args.steps
    kp_fwd_ms = timed(lambda: hp.ra.ra_attention_forward(qm, km, vm, scale=w.scale, out_dtype=torch.float32, mask=kpm))
    kp_bwd_ms = timed(lambda: hp.ra.ra_attention_backward(qm, km, vm, om, dom, rmm, rsm, ram, scale=w.scale, mask=kpm))
    if hp.ra.device_status() != "RA_OK":
        raise RuntimeError("masked attention: device status " + hp.ra.device_status())
    del kpm, om, rmm, rsm, ram

    # ra_softmax backward on the step's softmax workload (reported beside the step): x, the
    # forward's p, and a seeded dy; 16 B per element (x, p, dy read, dx written)
    xs, ps = hp.dev_in[4], hp.outs[4]
    dys = softmax_inputs(sw.rows, sw.cols, seed=sw.seed + 1, sigma=1.0).to(dev)
    dxs = torch.empty_like(dys)

    def softmax_bwd():
        code = hp.L.ra_softmax_bwd(_ptr(xs), _ptr(ps), _ptr(dys), _ptr(dxs), sw.rows, sw.cols, 0, st)
        if code != 0:
            raise RuntimeError("ra_softmax_bwd failed")
    hp.softmax(st)   # p for the timed x
    for _ in range(3):
        softmax_bwd()
    torch.cuda.synchronize(dev)
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(args.steps):
        softmax_bwd()
    b1.record(stream)
    torch.cuda.synchronize(dev)
    smb_ms = b0.elapsed_time(b1) / args.steps
    smb_bytes = 4.0 * x.numel() * 4
    del dys, dxs

    # ra_softmax with bf16 input and output on the same workload (4 B per element)
    xs16 = xs.to(torch.bfloat16)
    ys16 = torch.empty_like(xs16)

    def softmax_bf16():
        code = hp.L.ra_softmax_fwd(_ptr(xs16), _ptr(ys16), sw.rows, sw.cols, 1, st)
        if code != 0:
            raise RuntimeError("ra_softmax_fwd (bf16) failed")
    for _ in range(3):
        softmax_bf16()
    torch.cuda.synchronize(dev)
    b0.record(stream)
    for _ in range(args.steps):
        softmax_bf16()
    b1.record(stream)
    torch.cuda.synchronize(dev)
    sm16_ms = b0.elapsed_time(b1) / args.steps
    sm16_bytes = 2.0 * x.numel() * 2

    # bf16 ra_softmax backward: the bf16 x, its bf16 p, a bf16 dy; 8 B per element
    dy16 = softmax_inputs(sw.rows, sw.cols, seed=sw.seed + 1, sigma=1.0).to(dev).to(torch.bfloat16)
    dx16 = torch.empty_like(dy16)

    def softmax_bwd_bf16():
        code = hp.L.ra_softmax_bwd(_ptr(xs16), _ptr(ys16), _ptr(dy16), _ptr(dx16), sw.rows, sw.cols, 1, st)
        if code != 0:
            raise RuntimeError("ra_softmax_bwd (bf16) failed")
    for _ in range(3):
        softmax_bwd_bf16()
    torch.cuda.synchronize(dev)
    b0.record(stream)
    for _ in range(args.steps):
        softmax_bwd_bf16()
    b1.record(stream)
    torch.cuda.synchronize(dev)
    smb16_ms = b0.elapsed_time(b1) / args.steps
    smb16_bytes = 4.0 * x.numel() * 2
    del xs16, ys16, dy16, dx16

    # the RaAttention module at the page's example shape (dim 768, 12 heads, causal,
    # x [2, 128, 768], bf16): forward + backward through the module, seeded weights
    torch.manual_seed(0)
    mod = hp.ra.RaAttention(768, num_heads=12, causal=True).to(device=dev, dtype=torch.bfloat16)
    gx = torch.Generator().manual_seed(1)
    xm = torch.randn(2, 128, 768, generator=gx).to(dev, torch.bfloat16).requires_grad_(True)
    dym = torch.randn(2, 128, 768, generator=gx).to(dev, torch.bfloat16)

    def module_step():
        mod(xm).backward(dym)
    for _ in range(3):
        module_step()
    torch.cuda.synchronize(dev)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m0.record(torch.cuda.current_stream(dev))
    for _ in range(args.steps):
        module_step()
    m1.record(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    mod_ms = m0.elapsed_time(m1) / args.steps
    del mod, xm, dym

    # fp32-input attention at scale (the CUDA-core FFMA path the 2e-5 fp32 tolerance needs):
    # B1 H16 N4096 D128, non-causal, forward and backward, 3 timed calls each
    qf, kf, vf, dof = (t.to(dev) for t in attention_inputs(1, 16, 4096, 4096, 128, seed=11, dtype=torch.float32))

    def fp32_fwd():
        return hp.ra.ra_attention_forward(qf, kf, vf, causal=False, out_dtype=torch.float32)
    for _ in range(2):
        of, rmf, rsf, raf, _ = fp32_fwd()
    torch.cuda.synchronize(dev)
    m0.record(torch.cuda.current_stream(dev))
    for _ in range(3):
        of, rmf, rsf, raf, _ = fp32_fwd()
    m1.record(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    f32_fwd_ms = m0.elapsed_time(m1) / 3

    def fp32_bwd():
        return hp.ra.ra_attention_backward(qf, kf, vf, of, dof, rmf, rsf, raf, causal=False)
    fp32_bwd()
    torch.cuda.synchronize(dev)
    m0.record(torch.cuda.current_stream(dev))
    for _ in range(3):
        fp32_bwd()
    m1.record(torch.cuda.current_stream(dev))
    torch.cuda.synchronize(dev)
    f32_bwd_ms = m0.elapsed_time(m1) / 3
    if hp.ra.device_status() != "RA_OK":
        raise RuntimeError("fp32 attention component failed")
    f32_fwd_fl = attn_flops(1, 16, 4096, 4096, 128, False, False)
    f32_bwd_fl = attn_flops(1, 16, 4096, 4096, 128, False, True) - f32_fwd_fl
    # FFMA peak from the unit counts: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz
    ffma_peak = 152 * 128 * 2 * 2.07e9 / 1e12
    del qf, kf, vf, dof, of, rmf, rsf, raf

    # the two small configurations: the fp32 forward B1 H2 N128 D64 (scale 1/8) and the bf16
    # forward + backward B2 H12 N128 D64 causal (scale 1/8); latency-bound, times per call
    # through the binding (each call launches one or two tiny grids)
    w1 = ATTN_TINY_FP32
    q1, k1, v1 = (t.to(dev) for t in workload_inputs(w1))

    def tiny_fwd():
        return hp.ra.ra_attention_forward(q1, k1, v1, scale=w1.scale, causal=w1.causal, out_dtype=torch.float32)
    w3 = ATTN_MODULE_SHAPE
    q3, k3, v3, do3 = (t.to(dev) for t in workload_inputs(w3))

    def small_fwd_bwd():
        o3, rm3, rs3, ra3, _ = hp.ra.ra_attention_forward(q3, k3, v3, scale=w3.scale, causal=w3.causal,
                                                          out_dtype=torch.float32)
        hp.ra.ra_attention_backward(q3, k3, v3, o3, do3, rm3, rs3, ra3, scale=w3.scale, causal=w3.causal)

    def per_call_ms(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        m0.record(torch.cuda.current_stream(dev))
        for _ in range(n):
            fn()
        m1.record(torch.cuda.current_stream(dev))
        torch.cuda.synchronize(dev)
        return m0.elapsed_time(m1) / n
    tiny_ms = per_call_ms(tiny_fwd, max(args.steps, 20))
    small_ms = per_call_ms(small_fwd_bwd, max(args.steps, 20))
    if hp.ra.device_status() != "RA_OK":
        raise RuntimeError("small-configuration components failed")
    tiny_fl = attn_flops(w1.B, w1.H, w1.N, w1.N, w1.D, w1.causal, False)
    small_fl = attn_flops(w3.B, w3.H, w3.N, w3.N, w3.D, w3.causal, True)
    del q1, k1, v1, q3, k3, v3, do3

    peaks, peak_src = load_peaks()
    # every kernel here is timed in a loop of well under a second at the maximum SM clock
    # (the clocks entry of this line), so the burst figures are the denominators
    tc_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tc_sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bwd_tflops = bwd_fl / (med["ra_attention_bwd_ms"] * 1e-3) / 1e12
    fwd_tflops = fwd_fl / (med["ra_attention_fwd_ms"] * 1e-3) / 1e12
    sm_gbs = sm_bytes / (med["ra_softmax_ms"] * 1e-3) / 1e9
    n_qkvo = B * H * N * D
    # Algorithmic work per launch of each kernel of the step.  The backward's standard count
    # is five products (S recomputed, dP, dV, dK, dQ); the dK/dV kernel forms four of them
    # and the dQ kernel the fifth (its own recomputation of S and dP is counted nowhere).
    kern = {
        "ra_softmax_fwd_vec_kernel": ("hbm", sm_bytes, "4 B read + 4 B written per element"),
        "bf16_to_f16_kernel (fwd)": ("hbm", 4.0 * n_qkvo, "V: 2 B read + 2 B written per element"),
        "attn_fwd_tc_kernel": ("tensor", fwd_fl, "4 B H N^2 D FLOP (Q K^T and P V)"),
        "bf16_to_f16_kernel (bwd)": ("hbm", 16.0 * n_qkvo, "Q, K, V, dO: 2 B read + 2 B written per element"),
        "attn_bwd_dq_tc_kernel": ("tensor", 0.2 * bwd_fl, "2 B H N^2 D FLOP (dQ = dS K; its S and dP "
                                                         "recomputation is not counted)"),
        "attn_bwd_dkdv_tc_kernel": ("tensor", 0.8 * bwd_fl, "8 B H N^2 D FLOP (S^T, dP^T, dV, dK)"),
    }
    kernels = {}
    for name, (bound, work, what) in kern.items():
        ms = med[name]
        achieved = work / (ms * 1e-3) / (1e12 if bound == "tensor" else 1e9)
        peak = tc_burst if bound == "tensor" else hbm_peak
        kernels[name] = {"ms": ms, "bound": bound, "achieved": achieved, "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                         "frac": achieved / peak, "algorithmic": what}
    dominant = max(kernels, key=lambda k: kernels[k]["ms"])
    dk = kernels[dominant]
    traffic = traffic_from_profiles(dominant.replace(" (", "_").replace(")", ""))
    rl = {"bound": dk["bound"], "achieved": dk["achieved"], "peak": tc_burst if dk["bound"] == "tensor" else hbm_peak,
          "unit": dk["unit"], "frac": dk["frac"], "traffic": traffic, "kernel": dominant,
          "algorithmic": f"{kern[dominant][1]:.4e} {'FLOP' if dk['bound'] == 'tensor' else 'B'} per launch: "
                         f"{kern[dominant][2]}",
          "peak_source": f"{peak_src} ({'bf16 burst' if dk['bound'] == 'tensor' else 'HBM copy'}): the kernel runs "
                         f"{dk['ms']:.2f} ms per launch inside a {elapsed_ms / 1e3:.2f} s timed region"}
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded torch.randn (CPU generator), no dataset",
        "config": step_config(w, sw),
        "kernels": kernels,
        "components": {
            "ra_softmax": {"ms": med["ra_softmax_ms"], "GB_per_s": sm_gbs, "frac_hbm": sm_gbs / hbm_peak,
                           "frac_hbm_8000": sm_gbs / 8000.0},
            "ra_attention_fwd": {"ms": med["ra_attention_fwd_ms"], "TFLOP_per_s": fwd_tflops,
                                 "frac_bf16_burst": fwd_tflops / tc_burst,
                                 "tiles_visited": visited, "tiles_skipped": skipped,
                                 "skipped_fraction": (skipped / visited) if visited else None},
            "ra_attention_bwd": {"ms": med["ra_attention_bwd_ms"], "TFLOP_per_s": bwd_tflops,
                                 "frac_bf16_burst": bwd_tflops / tc_burst,
                                 "frac_bf16_sustained": bwd_tflops / tc_sustained},
            "ra_attention_keypad_half_b4h16n8192d128": {
                "fwd_ms": kp_fwd_ms, "bwd_ms": kp_bwd_ms,
                "note": "the step's attention with the second half of the keys masked for every query "
                        "(through the binding); every query tile's mask is a run of leading keys, so the "
                        "unmasked code runs over the first half of the keys: about half the work"},
            "ra_attention_fwd_causal_b4h16n8192d128": {"ms": causal_ms,
                                                       "TFLOP_per_s": causal_fl / (causal_ms * 1e-3) / 1e12,
                                                       "frac_bf16_burst": causal_fl / (causal_ms * 1e-3) / 1e12 / tc_burst},
            "ra_attention_fwd_fp32_b1h2n128d64": {
                "ms": tiny_ms, "TFLOP_per_s": tiny_fl / (tiny_ms * 1e-3) / 1e12,
                "note": "one tiny fp32 forward per call through the binding; latency-bound, no roofline claim"},
            "ra_attention_fwdbwd_bf16_b2h12n128d64_causal": {
                "ms": small_ms, "TFLOP_per_s": small_fl / (small_ms * 1e-3) / 1e12,
                "note": "forward + backward per call through the binding (24 heads of one 128-row tile); "
                        "latency-bound, no roofline claim"},
            "ra_softmax_bf16": {"ms": sm16_ms, "GB_per_s": sm16_bytes / (sm16_ms * 1e-3) / 1e9,
                                "frac_hbm": sm16_bytes / (sm16_ms * 1e-3) / 1e9 / hbm_peak,
                                "algorithmic": "4 B per element (bf16 read and written)"},
            "ra_softmax_bwd": {"ms": smb_ms, "GB_per_s": smb_bytes / (smb_ms * 1e-3) / 1e9,
                               "frac_hbm": smb_bytes / (smb_ms * 1e-3) / 1e9 / hbm_peak,
                               "algorithmic": "16 B per element (x, p, dy read; dx written)"},
            "ra_softmax_bwd_bf16": {"ms": smb16_ms, "GB_per_s": smb16_bytes / (smb16_ms * 1e-3) / 1e9,
                                    "frac_hbm": smb16_bytes / (smb16_ms * 1e-3) / 1e9 / hbm_peak,
                                    "algorithmic": "8 B per element (bf16 x, p, dy read; dx written)"},
            "ra_attention_module_b2n128d768h12_causal": {
                "ms_fwd_bwd": mod_ms, "tokens_per_s": 2 * 128 / (mod_ms * 1e-3),
                "note": "latency-bound (24 heads of one 128-row tile); no roofline claim"},
            "ra_attention_fp32_b1h16n4096d128": {
                "fwd_ms": f32_fwd_ms, "fwd_TFLOP_per_s": f32_fwd_fl / (f32_fwd_ms * 1e-3) / 1e12,
                "bwd_ms": f32_bwd_ms, "bwd_TFLOP_per_s": f32_bwd_fl / (f32_bwd_ms * 1e-3) / 1e12,
                "bound": "alu", "peak_TFLOP_per_s": ffma_peak,
                "fwd_frac": f32_fwd_fl / (f32_fwd_ms * 1e-3) / 1e12 / ffma_peak,
                "bwd_frac": f32_bwd_fl / (f32_bwd_ms * 1e-3) / 1e12 / ffma_peak,
                "note": "fp32 inputs, FFMA only (no TF32); counted FLOPs; peak = 152 SMs x 128 lanes x 2 x 2.07 GHz"},
        },
        "roofline": rl,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": hp.h2d_bytes(),
                "d2h_bytes_per_step": hp.d2h_bytes(), "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": 6 * args.steps,
        "gpu_launches_per_step": {"ra_softmax_fwd_vec_kernel": 1, "attn_fwd_tc_kernel": 1, "bf16_to_f16_kernel": 2,
                                  "attn_bwd_dq_tc_kernel": 1, "attn_bwd_dkdv_tc_kernel": 1},
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, desc = cpu_oracle_sample(w, sw, q, k, v, do, x)
        line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_threads(),
                                "kind": "oracle", "sample": desc, "seconds": dt}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The float64 CPU oracle on a bounded sample of the same workload, per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from rational_softmax_attention_gb300.inputs import ATTN_LONG_WIDE, RA_SOFTMAX_LONG_ROWS, softmax_inputs, workload_inputs
    w, sw = ATTN_LONG_WIDE, RA_SOFTMAX_LONG_ROWS
    q, k, v, do = workload_inputs(w)
    x = softmax_inputs(sw.rows, sw.cols, seed=sw.seed, sigma=sw.sigma)
    for _ in range(args.warmup):
        cpu_oracle_sample(w, sw, q, k, v, do, x, query_rows=256, softmax_rows=16, heads=1)
    total, flops, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = cpu_oracle_sample(w, sw, q, k, v, do, x, query_rows=256, softmax_rows=16, heads=1)
        total += dt
        flops += fl
    value = flops / total / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic: seeded torch.randn (CPU generator), no dataset",
        "config": step_config(w, sw),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_threads(), "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu part", "hardware")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def run_oracle_configs(max_heads):
    """The float64 oracle timed on this host's cores for each of the five workloads (inputs
    drawn before the clock starts).  Attention workloads time up to `max_heads` heads and
    scale linearly to all heads (the work is exactly linear in heads); ra_softmax times 2048
    of its 16384 rows and scales by rows.  One JSON line per workload."""
    import oracle
    from rational_softmax_attention_gb300.inputs import (ATTN_LONG_CAUSAL, ATTN_LONG_WIDE, ATTN_MODULE_SHAPE,
                                                         ATTN_TINY_FP32, RA_SOFTMAX_LONG_ROWS, softmax_inputs,
                                                         workload_inputs)
    base = {"cores": cpu_threads(), "cpu": cpu_model(), "kind": "oracle (float64 NumPy, materialised per head)"}
    for w in (ATTN_TINY_FP32, RA_SOFTMAX_LONG_ROWS, ATTN_MODULE_SHAPE, ATTN_LONG_CAUSAL, ATTN_LONG_WIDE):
        if w is RA_SOFTMAX_LONG_ROWS:
            rows = 2048
            xd = softmax_inputs(w.rows, w.cols, seed=w.seed, sigma=w.sigma)[:rows].double().numpy()
            t0 = time.perf_counter()
            oracle.ra_softmax(xd)
            dt = time.perf_counter() - t0
            print(json.dumps({"workload": w.name, "seconds_timed": dt, "timed": f"{rows} of {w.rows} rows",
                              "seconds_all": dt * w.rows / rows, **base}), flush=True)
            continue
        ts = workload_inputs(w)
        heads = [(b, h) for b in range(w.B) for h in range(w.H)][:max_heads]
        dt = 0.0
        for b, h in heads:
            qd, kd, vd = (t[b, h].double().numpy() for t in ts[:3])
            t0 = time.perf_counter()
            oracle.ra_attention_head_fwd(qd, kd, vd, w.scale, w.causal)
            if w.backward:
                oracle.ra_attention_head_bwd(qd, kd, vd, ts[3][b, h].double().numpy(), w.scale, w.causal)
            dt += time.perf_counter() - t0
        nh = w.B * w.H
        print(json.dumps({"workload": w.name, "seconds_timed": dt, "timed": f"{len(heads)} of {nh} heads",
                          "seconds_all": dt * nh / len(heads), "backward": w.backward, **base}), flush=True)


def run_profile_case():
    """A small fixed case for ncu captures: ra_softmax on fp32 [8192, 8192] and attention
    forward + backward at B2 H16 N8192 D128 bf16 (inputs ~0.3 GB, larger than L2), twice."""
    import torch

    import rational_softmax_attention_gb300 as ra
    from rational_softmax_attention_gb300.inputs import attention_inputs, softmax_inputs

    q, k, v, do = (t.cuda() for t in attention_inputs(2, 16, 8192, 8192, 128, seed=0, sigma_qk=3.0))
    x = softmax_inputs(8192, 8192, seed=1, sigma=4.0).cuda()
    for _ in range(2):
        ra.ra_softmax(x)
        o, rm, rs, rarg, _ = ra.ra_attention_forward(q, k, v, scale=128 ** -0.5, out_dtype=torch.float32)
        ra.ra_attention_backward(q, k, v, o, do, rm, rs, rarg, scale=128 ** -0.5)
    torch.cuda.synchronize()
    status = ra.device_status()
    print("profile case status", status)
    if status != "RA_OK":
        raise SystemExit(1)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing on the host")
    ap.add_argument("--profile-case", action="store_true",
                    help="run only the small fixed case used for ncu captures, then exit")
    ap.add_argument("--oracle-configs", type=int, metavar="MAX_HEADS", default=0,
                    help="time the float64 oracle on the host for each workload (up to MAX_HEADS heads), then exit")
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case()
        return
    if args.oracle_configs:
        run_oracle_configs(args.oracle_configs)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
