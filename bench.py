#!/usr/bin/env python3
"""Benchmark of the GB300 transposed-convolution library.

Default workload: the fused ConvTranspose3d + add + x*hardswish(x) in fp32,
x (128, 32, 16, 16, 16), w (32, 64, 3, 3, 3), k=3, s=2, p=1, op=1, bias, add
(128, 64, 32, 32, 32) -- the largest workload of the set (2.2 GB per step) --
inputs resident in HBM, one step = one forward pass over the whole batch
through the C ABI, at FP32 accuracy (CT_F32: the three-term tf32 split on the
tensor cores).  `--split2` runs the opt-in two-term bf16 split
(CT_F32_BF16X2) instead and says so in the line.

Prints ONE JSON line (rank 0).  `value` is throughput in GFLOP/s of
algorithmic work (2 x the multiply-adds whose tap lands inside the output),
summed over ranks; GB/s of algorithmic bytes (every tensor read or written
once) is reported beside it.  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.  `--table` prints one line per
workload (the five sizes of the workload set) for the roofline table.

Multi-GPU (torchrun): every rank runs the full workload on its own GPU
(independent replicas, weak scaling), barrier + synchronise around the
timed region, time = max over ranks, value = units of all ranks / time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEADLINE = "convT3d_add_hswish"
METRIC = "ConvTranspose fwd GFLOP/s (and GB/s) on 1 GB300; % of roofline vs CPU oracle"
L2_BYTES = 129 * 1024 * 1024
SMS = 152
FP32_LANES_PER_SM = 128


# ----------------------------------------------------------------------------- work model
def out_len(L, k, s, p, op, d):
    return (L - 1) * s - 2 * p + d * (k - 1) + op + 1


def landed_pairs(L_in, k, s, p, op, d):
    """Number of (input position, tap) pairs of one dimension whose target
    o = i*s - p + k*d lies inside [0, L_out)."""
    Lo = out_len(L_in, k, s, p, op, d)
    n = 0
    for kk in range(k):
        # i in [0, L_in) with 0 <= i*s - p + kk*d < Lo
        lo = max(0, -(-(p - kk * d) // s))
        hi = min(L_in - 1, (Lo - 1 + p - kk * d) // s)
        n += max(0, hi - lo + 1)
    return n


def work_model(cfg, N=None):
    """Algorithmic FLOPs (2 per landed multiply-add) and bytes (each tensor
    read or written once) of one forward pass."""
    N = cfg["N"] if N is None else N
    nd = cfg["nd"]
    pairs = 1
    Lo = []
    for d in range(nd):
        args = (cfg["L_in"][d], cfg["k"][d], cfg["stride"][d], cfg["padding"][d],
                cfg["output_padding"][d], cfg["dilation"][d])
        pairs *= landed_pairs(*args)
        Lo.append(out_len(*args))
    Cog = cfg["C_out"] // cfg["groups"]
    macs = N * cfg["C_in"] * Cog * pairs
    esz = 2 if cfg["dtype"] == "bf16" else 4
    x_b = N * cfg["C_in"] * int(np.prod(cfg["L_in"])) * esz
    w_b = cfg["C_in"] * Cog * int(np.prod(cfg["k"])) * esz
    y_e = N * cfg["C_out"] * int(np.prod(Lo))
    b_b = cfg["C_out"] * 4 if cfg["bias"] else 0
    add_b = y_e * 4 if cfg["add"] else 0
    return dict(flops=2 * macs, bytes=x_b + w_b + b_b + add_b + y_e * 4, x_bytes=x_b, w_bytes=w_b,
                bias_bytes=b_b, add_bytes=add_b, y_bytes=y_e * 4, out_shape=[N, cfg["C_out"]] + Lo)


# ----------------------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    except Exception:
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0,
                    source="fallback")


def fp32_alu_peak_tflops(sm_mhz):
    # FFMA: 128 FP32 lanes per SM, 2 FLOP per lane per clock
    return SMS * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # nvidia-smi takes a while to start: wait (bounded) for its first
            # sample, so that even a timed region shorter than the sampling
            # interval has samples right before and after it
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.005)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        n0 = len(self.lines)
        t0 = time.time()
        while len(self.lines) == n0 and time.time() - t0 < 0.5 and self.proc.poll() is None:
            time.sleep(0.005)             # one more sample, taken after the timed region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for_smi(local):
    """nvidia-smi -i accepts a UUID; torch's device index may differ from
    nvidia-smi's numbering when only some GPUs are visible."""
    try:
        import torch
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(local)


# ----------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value, ws):
    """Max of a float over ranks (identity without a process group)."""
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate(units_all_ranks, max_seconds):
    """Whole-job throughput: units of all ranks over the slowest rank's time."""
    return units_all_ranks / max_seconds if max_seconds > 0 else float("nan")


# ----------------------------------------------------------------------------- GPU arm
def _inputs_to_device(cfg_name, dev, pinned=False, batch=None):
    import torch
    t = workloads.config_inputs(cfg_name, N=batch)
    cfg = workloads.CONFIGS[cfg_name]
    host = {}
    if cfg["dtype"] == "bf16":
        host["x"] = torch.from_numpy(t["x_bits"].view(np.int16)).view(torch.bfloat16)
        host["w"] = torch.from_numpy(t["w_bits"].view(np.int16)).view(torch.bfloat16)
    else:
        host["x"] = torch.from_numpy(t["x"])
        host["w"] = torch.from_numpy(t["w"])
    host["bias"] = torch.from_numpy(t["bias"]) if t["bias"] is not None else None
    host["add"] = torch.from_numpy(t["add"]) if t["add"] is not None else None
    if cfg.get("layout", "cf") == "cl":
        # channels-last workloads store x (and add) as (N, spatial..., C)
        for k in ("x", "add"):
            if host[k] is not None:
                host[k] = host[k].movedim(1, -1).contiguous()
    if pinned:
        host = {k: (v.pin_memory() if v is not None else None) for k, v in host.items()}
    devt = {k: (v.to(dev) if v is not None else None) for k, v in host.items()}
    return host, devt


class Runner:
    """One forward pass of a workload through the C ABI, buffers pre-allocated."""

    def __init__(self, cfg_name, dev, batch=None, split2=False):
        import torch
        import transposed_convolution_convtranspose_gb300 as ct
        self.ct = ct
        self.cfg = dict(workloads.CONFIGS[cfg_name])
        if batch is not None:
            self.cfg["N"] = batch
            if self.cfg["add"]:
                self.cfg["out_shape"] = (batch,) + tuple(self.cfg["out_shape"][1:])
        self.name = cfg_name
        self.dev = dev
        self.host, self.d = _inputs_to_device(cfg_name, dev, pinned=True, batch=batch)
        wm = work_model(self.cfg)
        self.wm = wm
        self.cl = self.cfg.get("layout", "cf") == "cl"
        y_shape = list(wm["out_shape"])
        if self.cl:
            y_shape = [y_shape[0]] + y_shape[2:] + [y_shape[1]]
        self.y = torch.empty(y_shape, dtype=torch.float32, device=dev)
        self.y_host = torch.empty(y_shape, dtype=torch.float32).pin_memory()
        c = self.cfg
        self.split2 = bool(split2) and c["dtype"] != "bf16"
        self.dt = ct.CT_BF16 if c["dtype"] == "bf16" else (ct.CT_F32_BF16X2 if self.split2 else ct.CT_F32)
        if self.cl:
            args = (c["nd"], c["N"], c["C_in"], c["C_out"], c["L_in"], c["k"], c["groups"], c["stride"],
                    c["padding"], c["output_padding"], c["dilation"], self.dt)
            self.ws_bytes = ct.ct_workspace_size_cl(*args)
            self.path = ct.ct_path_cl(*args, c["add"])
        elif c["nd"] == 1:
            self.ws_bytes = ct.ct_workspace_size_1d(c["N"], c["C_in"], c["C_out"], c["L_in"][0], c["k"][0],
                                                    c["groups"], c["stride"][0], c["padding"][0],
                                                    c["output_padding"][0], c["dilation"][0], self.dt)
            self.path = ct.ct_path_1d(c["N"], c["C_in"], c["C_out"], c["L_in"][0], c["k"][0],
                                      c["groups"], c["stride"][0], c["padding"][0],
                                      c["output_padding"][0], c["dilation"][0], self.dt)
        elif c["nd"] == 2:
            self.ws_bytes = ct.ct_workspace_size_2d(c["N"], c["C_in"], c["C_out"], c["L_in"], c["k"],
                                                    c["groups"], c["stride"], c["padding"],
                                                    c["output_padding"], c["dilation"], self.dt)
            self.path = ct.ct_path_2d(c["N"], c["C_in"], c["C_out"], c["L_in"], c["k"], c["groups"],
                                      c["stride"], c["padding"], c["output_padding"], c["dilation"],
                                      self.dt, c["add"])
        else:
            self.ws_bytes = ct.ct_workspace_size_3d(c["N"], c["C_in"], c["C_out"], c["L_in"], c["k"],
                                                    c["groups"], c["stride"], c["padding"],
                                                    c["output_padding"], c["dilation"], self.dt)
            self.path = ct.ct_path_3d(c["N"], c["C_in"], c["C_out"], c["L_in"], c["k"], c["groups"],
                                      c["stride"], c["padding"], c["output_padding"], c["dilation"],
                                      self.dt, c["add"])
        self.ws = (torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
                   if self.ws_bytes else None)
        # kernels the library launches per forward pass on this path
        # (a prep / repack launch, then the GEMM kernel; the bf16 repack splits in
        # two when D*H*W is not a multiple of 8; channels last it is the weight
        # repack alone)
        in_sp = int(np.prod(c["L_in"]))
        self.launches_per_step = {"umma_bf16": 2 if (in_sp % 8 == 0 or self.cl) else 3, "tc3d_tf32x3": 2,
                                  "tc3dg_tf32x3": 2, "tc3s_tf32x3": 2, "tc3d_bf16x2": 2, "tc3dg_bf16x2": 2,
                                  "tc3s_bf16x2": 2}.get(self.path, 1)

    def forward(self, stream, d=None, y=None):
        c, ct = self.cfg, self.ct
        d = self.d if d is None else d
        y_out = self.y if y is None else y
        if self.cl:
            ct.ct_forward_cl(c["nd"], d["x"], d["w"], d["bias"], d["add"], y_out, c["N"], c["C_in"],
                             c["C_out"], c["L_in"], c["k"], c["groups"], c["stride"], c["padding"],
                             c["output_padding"], c["dilation"], self.dt, self.ws, self.ws_bytes, stream)
        elif c["nd"] == 1:
            ct.ct_forward_1d(d["x"], d["w"], d["bias"], y_out, c["N"], c["C_in"], c["C_out"],
                             c["L_in"][0], c["k"][0], c["groups"], c["stride"][0], c["padding"][0],
                             c["output_padding"][0], c["dilation"][0], self.dt, self.ws,
                             self.ws_bytes, stream)
        elif c["nd"] == 2:
            fwd = ct.ct_forward_2d_add_hswish if c["add"] else ct.ct_forward_2d
            extra = (d["add"],) if c["add"] else ()
            fwd(d["x"], d["w"], d["bias"], *extra, y_out, c["N"], c["C_in"], c["C_out"], c["L_in"],
                c["k"], c["groups"], c["stride"], c["padding"], c["output_padding"], c["dilation"],
                self.dt, self.ws, self.ws_bytes, stream)
        elif c["add"]:
            ct.ct_forward_3d_add_hswish(d["x"], d["w"], d["bias"], d["add"], y_out, c["N"],
                                        c["C_in"], c["C_out"], c["L_in"], c["k"], c["groups"],
                                        c["stride"], c["padding"], c["output_padding"],
                                        c["dilation"], self.dt, self.ws, self.ws_bytes, stream)
        else:
            ct.ct_forward_3d(d["x"], d["w"], d["bias"], y_out, c["N"], c["C_in"], c["C_out"],
                             c["L_in"], c["k"], c["groups"], c["stride"], c["padding"],
                             c["output_padding"], c["dilation"], self.dt, self.ws, self.ws_bytes,
                             stream)

    def h2d(self, d=None):
        d = self.d if d is None else d
        for k in ("x", "w", "bias", "add"):
            if self.host[k] is not None:
                d[k].copy_(self.host[k], non_blocking=True)

    def second_buffer_set(self):
        """Device inputs, device output and pinned host output of a second
        in-flight step (the end-to-end leg's double buffering)."""
        import torch
        d2 = {k: (torch.empty_like(v) if v is not None else None) for k, v in self.d.items()}
        y2 = torch.empty_like(self.y)
        yh2 = torch.empty(tuple(self.y.shape), dtype=torch.float32).pin_memory()
        return d2, y2, yh2

    def d2h(self):
        self.y_host.copy_(self.y, non_blocking=True)

    def h2d_bytes(self):
        return sum(v.numel() * v.element_size() for v in self.host.values() if v is not None)

    def d2h_bytes(self):
        return self.y.numel() * 4


def time_e2e(r, steps, ws):
    """End-to-end time of `steps` steps through the public API (max over ranks).
    Every step copies its inputs host -> device from pinned memory, runs the
    forward call and reads its output back into pinned memory, all inside the
    timed region.  Steps are pipelined like a streaming user would run them:
    two buffer sets, the copies in on one stream, the forward calls on a
    second, the copies out on a third, so step k's input copy and step k-1's
    output copy overlap step k's compute (events order each buffer's reuse).
    The clock is CUDA events: from the first copy in to the last copy out.
    (Splitting the copies over four streams per direction measured no faster:
    the copy out, ~180 GB/s into pinned host memory, bounds the step.)"""
    import torch
    sh, sc, sd = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    d2, y2, yh2 = r.second_buffer_set()
    bufs = [(r.d, r.y, r.y_host), (d2, y2, yh2)]
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run(nsteps):
        for k in range(nsteps):
            b = k % 2
            d, y, yh = bufs[b]
            if k >= 2:
                sh.wait_event(comp_done[b])     # step k-2 has consumed these inputs
            with torch.cuda.stream(sh):
                r.h2d(d)
            h2d_done[b].record(sh)
            sc.wait_event(h2d_done[b])
            if k >= 2:
                sc.wait_event(d2h_done[b])      # step k-2's output has been read back
            r.forward(sc, d, y)
            comp_done[b].record(sc)
            sd.wait_event(comp_done[b])
            with torch.cuda.stream(sd):
                yh.copy_(y, non_blocking=True)
            d2h_done[b].record(sd)

    torch.cuda.synchronize()
    run(2)                                      # warm-up of the streams and buffers
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(sh)
    run(steps)
    sd.wait_stream(sh)
    sd.wait_stream(sc)
    e1.record(sd)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    del d2, y2, yh2
    barrier(ws)
    return reduce_max(ms / 1e3, ws)


def time_steps(fn, steps, warmup, ws, flush=None, graph=True):
    """Device time of `steps` forward passes (CUDA events on the stream the
    work runs on), max over ranks.  With graph=True one forward pass (the
    library's whole launch sequence) is captured once in a CUDA graph and
    replayed, so host-side argument handling stays out of the device clock."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    run = fn
    if graph:
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()                       # one more eager pass on the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=s):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        run = g.replay
        run()
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    barrier(ws)
    torch.cuda.synchronize()
    if flush is None:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    else:
        ms = 0.0
        for _ in range(steps):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
    barrier(ws)
    torch.cuda.synchronize()
    return reduce_max(ms / 1e3, ws)


def dtype_of(cfg, path):
    """Arithmetic of the path: bf16 products with fp32 accumulation; fp32
    (FFMA, or the three-term tf32 split, whose error is that of fp32
    arithmetic); or the opt-in two-term bf16 split of fp32 operands."""
    if cfg["dtype"] == "bf16":
        return "bf16-in/f32-acc"
    if path.endswith("_bf16x2"):
        return "f32 operands as bf16 hi+lo pairs (opt-in, ~2^-16 per product)"
    return "f32"


def traffic_for(name, path):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    capture (profiles/traffic.json), or None when no capture matches or the
    kernel's source file has changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get("%s/%s" % (name, path))
        if e is None:
            return None
        src = os.path.join(ROOT, "transposed_convolution_convtranspose_gb300", "csrc", e["kernel_source"])
        with open(src, "rb") as f:
            if hashlib.sha1(f.read()).hexdigest() != e["source_sha1"]:
                return None
        return e.get("bytes_per_launch")
    except Exception:
        return None


def roofline(name, cfg, path, wm, sec, peaks):
    """Roofline entry for the dominant kernel of the step."""
    traffic = traffic_for(name, path)
    if cfg["dtype"] == "bf16" and path == "umma_bf16":
        achieved = wm["flops"] / sec / 1e12
        peak = peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peaks["source"] + " cuBLAS bf16 burst"}
    if path in ("tc1d_tf32x3", "tc3d_tf32x3", "tc3dg_tf32x3", "tc3s_tf32x3", "tc3d_bf16x2", "tc3dg_bf16x2",
                "tc3s_bf16x2"):
        # FP32 on the tensor cores.  The tf32x3 kernels do 3 tf32 products per
        # multiply-add at the tf32 rate (half the bf16 rate): the time of 6 bf16
        # products; the opt-in bf16x2 kernels 2 bf16 MMAs over twice the K: the
        # time of 4.  The roofline is the slower of that tensor time and the HBM
        # time of the algorithmic bytes.
        bf16_products = 4 if path.endswith("_bf16x2") else 6
        tensor_s = bf16_products * wm["flops"] / (peaks["bf16_tflops"] * 1e12)
        hbm_s = wm["bytes"] / (peaks["hbm_gbs"] * 1e9)
        if hbm_s >= tensor_s:
            achieved = wm["bytes"] / sec / 1e9
            return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                    "peak_source": peaks["source"] + " copy bandwidth",
                    "tensor_time_floor_us": round(tensor_s * 1e6, 1)}
        achieved = bf16_products * wm["flops"] / sec / 1e12
        peak = peaks["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1),
                "unit": "TFLOP/s (bf16-equivalent: %d bf16 products per multiply-add)" % bf16_products,
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peaks["source"] + " cuBLAS bf16 burst",
                "hbm_time_floor_us": round(hbm_s * 1e6, 1)}
    ai = wm["flops"] / wm["bytes"]
    alu_peak = fp32_alu_peak_tflops(peaks["sm_max_mhz"])
    ridge = alu_peak * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if ai >= ridge:
        achieved = wm["flops"] / sec / 1e12
        return {"bound": "alu", "achieved": round(achieved, 2), "peak": round(alu_peak, 2),
                "unit": "TFLOP/s", "frac": round(achieved / alu_peak, 4), "traffic": traffic,
                "peak_source": "152 SMs x 128 FP32 lanes x 2 FLOP x %.0f MHz max SM clock"
                % peaks["sm_max_mhz"]}
    achieved = wm["bytes"] / sec / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
            "peak_source": peaks["source"] + " copy bandwidth"}


def run_gpu_arm(args, ws, rank, local):
    import torch
    import transposed_convolution_convtranspose_gb300 as ct
    from transposed_convolution_convtranspose_gb300 import build
    build.build()
    ct.load()
    ct.ct_set_path_override(args.path_override)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = args.config
    r = Runner(name, dev, batch=args.batch, split2=args.split2)
    wm = r.wm
    big = wm["bytes"] > L2_BYTES
    flush_buf = None if big else torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    flush = None if big else (lambda: flush_buf.add_(1.0))

    sampler = ClockSampler(gpu_id_for_smi(local)) if rank == 0 else None
    if sampler:
        sampler.start()
    t_dev = time_steps(lambda: r.forward(torch.cuda.current_stream()), args.steps, args.warmup, ws,
                       flush, graph=not args.no_graph)
    clocks = sampler.stop() if sampler else None

    # end-to-end through the public API: H2D of every step's inputs from
    # pinned host memory, the forward call, D2H of its output -- all timed,
    # steps pipelined over two buffer sets and three streams
    e2e_steps = max(2, min(args.steps, 8))
    t_e2e = time_e2e(r, e2e_steps, ws)
    ct.ct_last_device_error(torch.cuda.current_stream())

    peaks = measured_peaks()
    sec = t_dev / args.steps
    units = wm["flops"]
    value = aggregate(units * ws * args.steps / 1e9, t_dev)        # GFLOP/s, all ranks
    gbs = aggregate(wm["bytes"] * ws * args.steps / 1e9, t_dev)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype_of(r.cfg, r.path),
        "data": "synthetic (seeded numpy PCG64; x~N(0,1), w~U(-b,b))",
        "config": {"workload": (name if args.batch is None else "%s (batch %d)" % (name, args.batch)) +
                   (" [CT_F32_BF16X2 opt-in]" if r.split2 else "") +
                   (" [path override %d]" % args.path_override if args.path_override else ""),
                   "desc": r.cfg["desc"], "global_batch": r.cfg["N"] * ws,
                   "parallelism": "replicas" if ws > 1 else "single",
                   "l2": ("inputs larger than L2 (%.0f MB per step)" % (wm["bytes"] / 1e6)) if big
                   else "L2 flushed between steps", "path": r.path,
                   "timing": "CUDA graph replay" if not args.no_graph else "eager calls"},
        "gbps": round(gbs, 1),
        "roofline": roofline(name if args.batch is None else name + "@N%d" % args.batch,
                             r.cfg, r.path, wm, sec, peaks),
        "e2e": {"value": round(aggregate(units * ws * e2e_steps / 1e9, t_e2e), 1), "unit": "GFLOP/s",
                "h2d_bytes_per_step": r.h2d_bytes(), "d2h_bytes_per_step": r.d2h_bytes(),
                "steps": e2e_steps, "ms_per_step": round(t_e2e / e2e_steps * 1e3, 3),
                "schedule": "pinned-host copies in, forward call, copies out on three streams, "
                            "two buffer sets (step k's copies overlap its neighbours' work)"},
        "gpu_launches": r.launches_per_step * args.steps,
        "clocks": clocks,
    }
    return res, r


# ----------------------------------------------------------------------------- CPU oracle
def _slice_cfg(cfg, frac, nb=1):
    """The workload with batch nb and its outermost spatial input extent cut to
    a fraction (same channels, kernel, stride, padding, dilation)."""
    c = dict(cfg)
    L = list(cfg["L_in"])
    L[0] = max(1, int(round(L[0] * frac)))
    c["L_in"] = tuple(L)
    c["N"] = nb
    return c


def _oracle_run(cfg, t, threads=None):
    """The oracle on one sample: the single-threaded parity oracle
    (threads=None) or the same scatter definition on `threads` host threads."""
    import oracle
    kw = dict(stride=tuple(cfg["stride"]), padding=tuple(cfg["padding"]),
              output_padding=tuple(cfg["output_padding"]), dilation=tuple(cfg["dilation"]),
              groups=cfg["groups"])
    if threads is None:
        y = oracle.conv_transpose(t["x"], t["w"], t["bias"], **kw)
    else:
        y = oracle.conv_transpose_mt(t["x"], t["w"], t["bias"], threads=threads, **kw)
    if cfg["add"]:
        y = oracle.add_hswish(y, t["add"])
    return y


def _sample_inputs(cfg, seed):
    x_shape = (cfg["N"], cfg["C_in"]) + tuple(cfg["L_in"])
    w_shape = (cfg["C_in"], cfg["C_out"] // cfg["groups"]) + tuple(cfg["k"])
    add_shape = None
    if cfg["add"]:
        add_shape = tuple(work_model(cfg)["out_shape"])
    return workloads.make_tensors(seed, x_shape, w_shape, cfg["bound"],
                                  bias_len=cfg["C_out"] if cfg["bias"] else None,
                                  add_shape=add_shape, dtype=cfg["dtype"])


def oracle_sample_plan(name, seconds, threads=None):
    """The sample the oracle (single-threaded, or on `threads` threads)
    finishes in about `seconds`: a fraction of one batch item, or as many
    whole batch items as fit (calibrated on a 1/64 slice of one item)."""
    import oracle
    oracle.build_oracle()
    oracle.build_oracle_mt()
    cfg = workloads.CONFIGS[name]
    small = _slice_cfg(cfg, 1.0 / 64)
    part = small["L_in"][0] / cfg["L_in"][0]       # the slice actually cut (at least one plane)
    t = _sample_inputs(small, cfg["seed"])
    t0 = time.perf_counter()
    _oracle_run(small, t, threads)
    dt = max(time.perf_counter() - t0, 1e-4)
    items = seconds * part / dt
    if items >= 2:
        # a slice that fits in cache runs faster than a whole item: time one item
        one = _slice_cfg(cfg, 1.0, 1)
        t = _sample_inputs(one, cfg["seed"])
        t0 = time.perf_counter()
        _oracle_run(one, t, threads)
        items = seconds / max(time.perf_counter() - t0, 1e-4)
    if items >= 2:
        nb = int(min(cfg["N"], items))
        return _slice_cfg(cfg, 1.0, nb), float(nb)
    frac = min(1.0, max(1.0 / 64, items))
    return _slice_cfg(cfg, frac), frac


def oracle_time(scfg, name, threads=None):
    """Run the oracle once on the sampled workload; returns (GFLOP/s of
    algorithmic work, seconds)."""
    t = _sample_inputs(scfg, workloads.CONFIGS[name]["seed"])
    t0 = time.perf_counter()
    _oracle_run(scfg, t, threads)
    sec = time.perf_counter() - t0
    return work_model(scfg)["flops"] / sec / 1e9, sec


def sample_desc(scfg, name, frac, threads=None):
    how = ("single-threaded C oracle in float64" if threads is None else
           "the oracle's scatter definition in float64 on %d host threads (C, pthreads, one output slice "
           "(n, oc) per task)" % threads)
    N = workloads.CONFIGS[name]["N"]
    if scfg["N"] > 1:
        what = "batch %d of %s at full spatial size (%d of its %d batch items)" % (scfg["N"], name, scfg["N"], N)
    else:
        what = ("batch 1 of %s with the outermost input extent cut to %s (%.3f of one batch item of %d)"
                % (name, tuple(scfg["L_in"]), frac, N))
    return "%s, %s" % (what, how)


def cpu_baseline(name, seconds):
    """The CPU baseline: the oracle's definition on every host core, with the
    single-threaded parity oracle beside it, each on a bounded sample."""
    import oracle
    cores = oracle.host_cores()
    scfg, frac = oracle_sample_plan(name, seconds, threads=cores)
    v, sec = oracle_time(scfg, name, threads=cores)
    scfg1, frac1 = oracle_sample_plan(name, seconds)
    v1, sec1 = oracle_time(scfg1, name)
    return {"value": round(v, 4), "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
            "sample": sample_desc(scfg, name, frac, cores), "seconds": round(sec, 2),
            "hardware_concurrency": os.cpu_count(),
            "single_core": {"value": round(v1, 4), "unit": "GFLOP/s", "cores": 1,
                            "sample": sample_desc(scfg1, name, frac1), "seconds": round(sec1, 2)}}


def run_reference_arm(args):
    """The CPU oracle as the reference arm: every step is one bounded sample,
    the oracle's definition on every host core."""
    import oracle
    cfg = workloads.CONFIGS[args.config]
    cores = oracle.host_cores()
    per_step = max(0.2, min(20.0, args.ref_seconds / (args.steps + args.warmup)))
    scfg, frac = oracle_sample_plan(args.config, per_step, threads=cores)
    for _ in range(args.warmup):
        oracle_time(scfg, args.config, threads=cores)
    runs = [oracle_time(scfg, args.config, threads=cores) for _ in range(args.steps)]
    tot = sum(s for _, s in runs)
    value = work_model(scfg)["flops"] * len(runs) / tot / 1e9
    desc = sample_desc(scfg, args.config, frac, cores)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / len(runs) * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": args.config, "desc": cfg["desc"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc + ", per step", "hardware_concurrency": os.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": "GFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE, choices=list(workloads.CONFIGS))
    ap.add_argument("--table", action="store_true", help="one line per workload")
    ap.add_argument("--path-override", type=int, default=0,
                    help="library path override: 0 automatic, 1 generic kernel, 2 no FP32 tensor-core path")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small cases for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls instead of a CUDA graph")
    ap.add_argument("--split2", action="store_true",
                    help="fp32 workloads with the opt-in two-term bf16 split (CT_F32_BF16X2)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="total oracle time budget of the reference arm")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3

    ws, rank, local = dist_env()
    if args.impl == "reference":
        # the oracle runs on rank 0 only; other ranks exit without work
        if rank == 0:
            print(json.dumps(run_reference_arm(args)), flush=True)
        return 0

    if ws > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")

    if args.table:
        import torch
        for name in workloads.CONFIG_ORDER:
            # every workload at its default arithmetic; the FP32 tensor-core
            # workloads a second time with the opt-in two-term bf16 split
            for split2 in (False, True):
                a2 = argparse.Namespace(**vars(args))
                a2.config = name
                a2.split2 = split2
                res, r = run_gpu_arm(a2, ws, rank, local)
                has_opt_in = r.path in ("tc3d_tf32x3", "tc3dg_tf32x3")
                del r
                torch.cuda.empty_cache()
                if rank == 0:
                    print(json.dumps(res), flush=True)
                if not has_opt_in:
                    break
            if name in ("convT3d_s3_disjoint", "convT3d_s3_k5"):
                # the generic gather kernel these shapes took before, for comparison
                a2 = argparse.Namespace(**vars(args))
                a2.config = name
                a2.path_override = 1
                res, r = run_gpu_arm(a2, ws, rank, local)
                del r
                torch.cuda.empty_cache()
                if rank == 0:
                    print(json.dumps(res), flush=True)
                ct_mod = __import__("transposed_convolution_convtranspose_gb300")
                ct_mod.ct_set_path_override(0)
        return 0

    res, r = run_gpu_arm(args, ws, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.config, args.cpu_seconds)
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
