#!/usr/bin/env python
"""Benchmark of the im2win hot path on GB300.

One step runs every operation of the path once over one batch of the cv1
layer of Table I of "Enabling Memory-efficient Im2win Convolution with
Multi-precision Support on GPU CUDA and Tensor Cores" (N=128, C_i=3, 227x227,
C_o=96, 11x11, stride 4), in fp16 and fp32, with seeded synthetic inputs:

  1. im2win transform, fp16             (x16 -> win16)
  2. tensor-core conv from the window   (win16, w16 -> out16; filter re-layout + tcgen05 kernel)
  3. fused tensor-core conv             (x16, w16 -> out16f; filter re-layout + tcgen05 kernel)
  4. im2win transform, fp32             (x32 -> win32)
  5. CUDA-core conv from the window     (win32, w32 -> out32; filter re-layout + FFMA kernel)

value = conv FLOPs of the step (3 x 2*N*C_o*H_o*W_o*C_i*H_f*W_f) / step time, in TFLOP/s,
summed over ranks (each rank runs its own batch: weak scaling, no collective on
the data path). Inputs are resident in HBM when the timed region starts; L2 is
flushed (a 512 MB write) between timed steps, outside the timed region.

e2e = the same FLOPs per step through the same API calls when every step also
copies its inputs from pinned host memory and its outputs back; consecutive
steps are pipelined over two device buffer sets and separate copy streams.

`--layout nhwc` runs the same step on channels-last tensors (x[N][H_i][W_i][C_i],
win[N][H_o][W_i*H_f][C_i], out[N][H_o][W_o][C_o]) through the *_nhwc calls.

`--impl reference` times the CPU oracle (plain fp64 C, OpenMP) on a bounded
sample of the same workload instead.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of each
# kernel on this workload, from one ncu capture of the current kernel source
# (summaries under profiles/); a kernel absent here has no capture of its
# current version.
DRAM_TRAFFIC: dict = {
    # conv_f32_kernel<96,6,16,3,2,0,0,0>, cv1: 211.1 MB read + 106.3 MB written
    # (profiles/conv_f32_kernel_cv1.md)
    ("cv1", "conv_f32_window_f32"): 317.4e6,
}

METRIC = "im2win conv TFLOPS and % of dense peak per layer shape; workspace bytes"
UNIT = "TFLOP/s"
SMS = 152


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "sm_max_mhz": float(d.get("sm_max_mhz", 2070.0)), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0, "source": "fallback"}


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.out = os.path.join("/tmp", f"im2win_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.out, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.out) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.unlink(self.out)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def max_over_ranks(values, dist_mod=None, device=None):
    """Each value's maximum over the ranks of the process group (the values
    themselves when there is no group): the job's time is its slowest rank's."""
    if dist_mod is None:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tflops(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs its own batch (weak scaling), all in
    the time of the slowest rank."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def conv_flops(layer) -> float:
    ho, wo = layer.out_hw
    return 2.0 * layer.N * layer.C_o * ho * wo * layer.C_i * layer.H_f * layer.W_f


def workload_str(layer) -> str:
    pd = "" if layer.plain else f", padding {layer.pad[0]}x{layer.pad[1]}, dilation {layer.dil[0]}x{layer.dil[1]}"
    return (f"{layer.name}: N={layer.N}, C_i={layer.C_i}, {layer.H_i}x{layer.W_i}, C_o={layer.C_o}, "
            f"{layer.H_f}x{layer.W_f}, stride {layer.s_h}x{layer.s_w}{pd}; {' and '.join(layer.dtypes)}")


class OracleSampler:
    """The oracle as it stands (im2win transform + fp64 direct conv), one image
    at a time on the leading images of the batch, the layer's dtypes alternating
    (each rounded to its dtype, then widened exactly). Inputs are drawn once."""

    def __init__(self, layer, n_images=8):
        import oracle
        from memory_efficient_cnn_gb300 import workloads as wl

        oracle.build()
        self.oracle, self.layer = oracle, layer
        self.inputs = []
        for d in layer.dtypes:
            x, w = wl.make_inputs(layer, d, n_images=n_images)
            self.inputs.append((x.double().numpy(), w.double().numpy()))
        self.i = 0
        self.per_img = conv_flops(layer) / layer.N

    def run(self, budget_s: float, max_images: int):
        """Images until `budget_s` of oracle time is spent (at least one)."""
        L, done, t_total = self.layer, 0, 0.0
        while (t_total < budget_s or done == 0) and done < max_images:
            x, w = self.inputs[self.i % len(self.inputs)]
            n = (self.i // len(self.inputs)) % x.shape[0]
            xd = np.ascontiguousarray(x[n:n + 1])
            t0 = time.perf_counter()
            if L.plain:
                self.oracle.im2win(xd, L.H_f, L.s_h)
                self.oracle.conv_direct(xd, w, (L.s_h, L.s_w))
            else:
                st = (L.s_h, L.s_w)
                self.oracle.im2win_pd(xd, w.shape, st, L.pad, L.dil)
                self.oracle.conv_direct_pd(xd, w, st, L.pad, L.dil)
            t_total += time.perf_counter() - t0
            done += 1
            self.i += 1
        return done, t_total

    def threads(self) -> int:
        return self.oracle.num_threads()


def run_reference(args, layer, rank, world):
    if rank != 0:
        return
    # each step: the oracle on a bounded sample of images of the workload
    smp = OracleSampler(layer)
    steps = []
    for s in range(args.warmup + args.steps):
        imgs, t = smp.run(budget_s=0.5, max_images=32)
        if s >= args.warmup:
            steps.append((imgs, t))
    tot_t = sum(t for _, t in steps)
    tot_imgs = sum(i for i, _ in steps)
    value = smp.per_img * tot_imgs / tot_t / 1e12
    sample = (f"{tot_imgs / len(steps):.1f} images of {layer.name} per step on average (im2win "
              f"transform + fp64 direct conv per image; {'/'.join(layer.dtypes)}-rounded inputs "
              f"alternate), a step ends after 32 images or 0.5 s of oracle time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / len(steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_str(layer), "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": smp.threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layer", default="cv1",
                    help="workload: cv1 (default, the headline) or another layer of the parity set")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the cpu_baseline (0 disables it)")
    ap.add_argument("--layout", choices=["nchw", "nhwc"], default="nchw",
                    help="tensor layout of input, window tensor and output")
    ap.add_argument("--batch", type=int, default=0,
                    help="images per step (default: the layer's batch); smaller batches keep "
                         "profiler captures small")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from memory_efficient_cnn_gb300 import workloads as wl

    layers = {l.name: l for l in wl.ALL + wl.PADDED}
    if args.layer not in layers:
        ap.error(f"--layer must be one of {sorted(layers)}")
    layer = layers[args.layer]
    if args.batch < 0:
        ap.error("--batch must be positive")
    batch_changed = args.batch > 0 and args.batch != layer.N
    if batch_changed:
        layer = layer.with_batch(args.batch)
    rank, world, local = _dist()
    if args.impl == "reference":
        run_reference(args, layer, rank, world)
        return

    import torch

    import memory_efficient_cnn_gb300 as mec

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    mec.lib()  # fail loudly if the library is missing

    # cpu baseline first (rank 0, N=1 only): before any other GPU work is queued
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        smp = OracleSampler(layer)
        imgs, t = smp.run(budget_s=args.cpu_budget, max_images=10 ** 9)
        cpu = {"value": smp.per_img * imgs / t / 1e12, "unit": UNIT, "cores": smp.threads(),
               "kind": "oracle",
               "sample": f"{imgs} images of {layer.name} (im2win transform + fp64 direct conv of the "
                         f"{'/'.join(layer.dtypes)} inputs, alternating), {t:.1f} s"}

    stride = (layer.s_h, layer.s_w)
    shp = layer.shape_args
    N, C_i, H_i, W_i, C_o, H_f, W_f, s_h, s_w = shp
    H_o, W_o = layer.out_hw
    W_p = W_i + 2 * layer.pad[1]  # window row: W_p*H_f elements
    pdargs = (*shp, layer.pad[0], layer.pad[1], layer.dil[0], layer.dil[1])

    # one step: per dtype, the transform, the conv from the window tensor and
    # (fp16/bf16) the fused conv; fp32 runs on the CUDA cores
    cl = args.layout == "nhwc"
    sfx = "_nhwc" if cl else ""
    host_in = []
    for d in layer.dtypes:
        xh, wh = wl.make_inputs(layer, d)
        host_in += [xh.permute(0, 2, 3, 1).contiguous() if cl else xh, wh]

    def make_set():
        """Device buffers of one step (inputs, window tensors, outputs, workspaces)
        and its calls through the public API."""
        ops, dev_in, outs = [], [], []
        for di, d in enumerate(layer.dtypes):
            add_dtype_ops(ops, dev_in, outs, d, host_in[2 * di], host_in[2 * di + 1])
        return ops, dev_in, outs

    def add_dtype_ops(ops, dev_in, outs, d, xc, wc):
        tdt = wl.DTYPES[d]
        x, w = xc.to(dev), wc.to(dev)
        dev_in += [x, w]
        nchw = (N, C_i, H_i, W_i)
        if cl:
            win = torch.empty((N, H_o, W_p * H_f, C_i), dtype=tdt, device=dev)
            out_w = torch.empty((N, H_o, W_o, C_o), dtype=tdt, device=dev)
        else:
            win = torch.empty((N, C_i, H_o, W_p * H_f), dtype=tdt, device=dev)
            out_w = torch.empty((N, C_o, H_o, W_o), dtype=tdt, device=dev)
        if not layer.plain:
            # padding / dilation: the *_ex calls, layout as an argument
            lo = mec.NHWC if cl else mec.NCHW
            dc = mec._binding._DTYPE[tdt]
            ws = torch.empty(mec.im2win_workspace_size_ex(mec.OP_CONV, *pdargs, lo, dc), dtype=torch.uint8,
                             device=dev)
            wsf = torch.empty(mec.im2win_workspace_size_ex(mec.OP_CONV_FUSED, *pdargs, lo, dc),
                              dtype=torch.uint8, device=dev)
            tr = lambda x, win: mec.im2win_transform_ex(x, win, *pdargs, lo)
            cv = lambda win, w, o, ws: mec.im2win_conv_ex(win, w, o, ws, *pdargs, lo)
            cvf = lambda x, w, o, ws: mec.im2win_conv_fused_ex(x, w, o, ws, *pdargs, lo)
        else:
            if cl:
                tr0, cv0, cvf0 = mec.im2win_transform_nhwc, mec.im2win_conv_nhwc, mec.im2win_conv_fused_nhwc
                op_w, op_f = mec.OP_CONV_NHWC, mec.OP_CONV_FUSED_NHWC
            else:
                tr0, cv0, cvf0 = mec.im2win_transform, mec.im2win_conv, mec.im2win_conv_fused
                op_w, op_f = mec.OP_CONV, mec.OP_CONV_FUSED
            ws = mec.workspace(op_w, nchw, w.shape, stride, tdt, dev)
            wsf = mec.workspace(op_f, nchw, w.shape, stride, tdt, dev)
            tr = lambda x, win, tr0=tr0: tr0(x, win, C_o, H_f, W_f, s_h, s_w)
            cv = lambda win, w, o, ws, cv0=cv0: cv0(win, w, o, ws, *shp)
            cvf = lambda x, w, o, ws, cvf0=cvf0: cvf0(x, w, o, ws, s_h, s_w)
        ops.append((f"transform_{d}{sfx}", d, "transform",
                    lambda x=x, win=win, tr=tr: tr(x, win),
                    {"win_bytes": win.numel() * win.element_size()}))
        kind = "conv_f32" if d == "f32" else "conv_tc"
        ops.append((f"{kind}_window_{d}{sfx}", d, "window",
                    lambda win=win, w=w, o=out_w, ws=ws, cv=cv: cv(win, w, o, ws),
                    {"ws_bytes": ws.numel()}))
        outs.append(out_w)
        if d != "f32":
            out_f = torch.empty_like(out_w)
            ops.append((f"conv_tc_fused_{d}{sfx}", d, "fused",
                        lambda x=x, w=w, o=out_f, ws=wsf, cvf=cvf: cvf(x, w, o, ws),
                        {"ws_bytes": wsf.numel()}))
            outs.append(out_f)

    ops, dev_in, outs = make_set()
    names = [o[0] for o in ops]
    n_ops = len(ops)
    n_convs = sum(1 for o in ops if o[2] != "transform")
    LAUNCHES_PER_STEP = sum(1 if o[2] == "transform" else 2 for o in ops)  # conv: re-layout + kernel
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None):
        for i, op in enumerate(ops):
            if evs:
                evs[i].record(stream)
            op[3]()
        if evs:
            evs[n_ops].record(stream)

    for _ in range(args.warmup):
        step()
        flush.zero_()
    torch.cuda.synchronize(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ops + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)
    for k in range(args.steps):
        step(ev[k])
        flush.zero_()
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if dist:
        dist.barrier()
    per = [[ev[k][i].elapsed_time(ev[k][i + 1]) for i in range(n_ops)] for k in range(args.steps)]
    step_ms = sum(sum(p) for p in per)
    kern_ms = [sum(p[i] for p in per) / args.steps for i in range(n_ops)]

    # ---- end to end through the public API from pinned host buffers: every step
    # copies its inputs in, runs the step and copies its outputs out. Steps are
    # pipelined over two device buffer sets and three streams (inputs of step k+1
    # and outputs of step k-1 move while step k computes), as a serving loop would;
    # the timed region spans all K steps, from the first input copy to the last
    # output copy.
    h_in = [t.pin_memory() for t in host_in]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    sets = [(ops, dev_in, outs), make_set()]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(nsteps, start=None):
        if start is not None:
            s_in.wait_event(start)
        for k in range(nsteps):
            b = k % 2
            set_ops, set_in, set_outs = sets[b]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(ev_done[b])  # step k-2 has read this set's inputs
                for d_, h in zip(set_in, h_in):
                    d_.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if k >= 2:
                stream.wait_event(ev_out[b])  # this set's outputs of step k-2 are out
            for op in set_ops:
                op[3]()
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                for h, d_ in zip(h_out, set_outs):
                    h.copy_(d_, non_blocking=True)
                ev_out[b].record(s_out)
        stream.wait_event(ev_out[(nsteps - 1) % 2])

    e2e_run(3)
    torch.cuda.synchronize(dev)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    e2e_run(args.steps, e_start)
    e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e_start.elapsed_time(e_end)

    if dist:
        step_ms, e2e_ms = max_over_ranks([step_ms, e2e_ms], dist, dev)
        dist.destroy_process_group()
    if rank != 0:
        return

    f = conv_flops(layer)
    ms = step_ms / args.steps
    value = job_tflops(world, n_convs * f, ms)
    e2e_value = job_tflops(world, n_convs * f, e2e_ms / args.steps)
    pk = _peaks()
    fp32_peak = SMS * 128 * 2 * pk["sm_max_mhz"] * 1e6 / 1e12  # FFMA lanes x 2 flop x clock
    # dense fp16/bf16 tcgen05 rate of the hardware: 4096 MAC per clock per SM
    # (8192 flop) at the maximum SM clock; cuBLAS's measured figure (the contract's
    # `peak`) sits below it
    mma_peak = SMS * 8192 * pk["sm_max_mhz"] * 1e6 / 1e12
    esz = {"f16": 2, "bf16": 2, "f32": 4}
    x_b = {d: N * C_i * H_i * W_i * esz[d] for d in esz}
    win_b = {d: N * C_i * H_o * W_p * H_f * esz[d] for d in esz}
    out_b = {d: N * C_o * H_o * W_o * esz[d] for d in esz}
    w_b = {d: C_o * C_i * H_f * W_f * esz[d] for d in esz}
    col_b = {d: N * C_i * H_f * W_f * H_o * W_o * esz[d] for d in esz}
    kernels = {}
    for i, (name, d, kind, _, extra) in enumerate(ops):
        t_s = kern_ms[i] * 1e-3
        if kind == "transform":
            byts = x_b[d] + win_b[d]
            kernels[name] = {"ms": kern_ms[i], "bound": "hbm", "achieved": byts / t_s / 1e9,
                             "peak": pk["hbm_gbs"], "unit": "GB/s", "alg_bytes": byts}
        elif d == "f32":
            kernels[name] = {"ms": kern_ms[i], "bound": "alu", "achieved": f / t_s / 1e12,
                             "peak": fp32_peak, "unit": "TFLOP/s", "flops": f}
        else:
            byts = (win_b[d] if kind == "window" else x_b[d]) + w_b[d] + out_b[d]
            tc_peak = pk["bf16_tflops"]
            hbm_cap = f / byts * pk["hbm_gbs"] * 1e9 / 1e12
            bound = "tensor" if tc_peak < hbm_cap else "hbm"
            kernels[name] = {"ms": kern_ms[i], "bound": bound, "achieved": f / t_s / 1e12,
                             "peak": min(tc_peak, hbm_cap), "unit": "TFLOP/s", "flops": f,
                             "alg_bytes": byts, "tensor_peak_frac": f / t_s / 1e12 / tc_peak,
                             "tcgen05_peak_frac": f / t_s / 1e12 / mma_peak}
        kernels[name]["frac"] = kernels[name]["achieved"] / kernels[name]["peak"]
        if "ws_bytes" in extra:
            kernels[name]["workspace_bytes"] = extra["ws_bytes"]
    workspace = {}
    for d in layer.dtypes:
        ws_conv = kernels[f"{'conv_f32' if d == 'f32' else 'conv_tc'}_window_{d}{sfx}"]["workspace_bytes"]
        workspace[f"two_step_{d}"] = win_b[d] + ws_conv
        if d != "f32":
            workspace[f"fused_{d}"] = kernels[f"conv_tc_fused_{d}{sfx}"]["workspace_bytes"]
        workspace[f"im2col_{d}"] = col_b[d]
    dom = max(kernels, key=lambda k: kernels[k]["ms"])
    dk = kernels[dom]
    # the captured traffic is that of the layer's own batch
    traffic = None if batch_changed else DRAM_TRAFFIC.get((layer.name, dom))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "+".join(layer.dtypes), "data": "synthetic",
        "config": {"workload": workload_str(layer), "layout": "NHWC" if cl else "NCHW",
                   "step": ", ".join(names),
                   "parallelism": f"replicas x{world}", "l2": "flushed between steps (512 MB write)"},
        "roofline": {"kernel": dom, "bound": dk["bound"], "achieved": dk["achieved"],
                     "peak": dk["peak"], "unit": dk["unit"], "frac": dk["frac"],
                     "traffic": traffic,
                     "peak_source": "fp32 FFMA: 152 SMs x 128 lanes x 2 x max SM clock"
                     if dk["bound"] == "alu" else pk["source"]},
        "kernels": kernels,
        "workspace_bytes": workspace,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "peaks": dict(pk, tcgen05_dense_tflops=mma_peak,
                      tcgen05_source="152 SMs x 8192 dense fp16/bf16 flop/clk x max SM clock; "
                                     "tensor_peak_frac is of the measured cuBLAS bf16 figure, "
                                     "tcgen05_peak_frac of this one"),
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
