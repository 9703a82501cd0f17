"""Benchmark of the fused conv + BN + activation hot path on GB300.

Default workload (N=1): the depthwise 3x3 + BN + ReLU layer, NHWC fp32,
x = [64, 56, 56, 384] ~ N(0,1), at stride 1 and stride 2; one step = both
launches over the batch.  ``value`` is algorithmic HBM bytes per second
(input + output + weights + scale/bias, per workloads.py) over the timed
steps, whole job (all ranks).  Other workloads (``--workload``) measure the
dense 3x3 sweep, the DepthwiseMNIST forward, the YOLO-style chain and the
preprocess -> stem pipeline.

Multi-GPU (torchrun): images are independent, so every rank runs its own
batch (weak scaling, no data-path collective); ranks meet only at the
barriers around the timed region and for the max-time / sum-units reduction.

``--impl reference`` times the CPU oracle (the plain fp64 reference) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor rates


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------ clocks sampler
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes) every ~1 ms on a
    background thread while the timed region runs.  Read-only: changes no setting."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, device_index: int):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        self.samples = []
        self.ok = False
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            got = False
            try:
                uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
                got = lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                got = False
            if not got:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[device_index]) if vis and vis.split(",")[0].isdigit() else device_index
                got = lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) == 0
            if not got:
                return
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))
            self.lib, self.h, self.max_mhz = lib, h, mx.value
            self.ok = True
        except OSError:
            return

    def _loop(self):
        c, r = self.ctypes.c_uint(), self.ctypes.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ctypes.byref(c)) == 0 and \
                    self.reason_fn(self.h, self.ctypes.byref(r)) == 0:
                self.samples.append((c.value, r.value))
            time.sleep(0.001)

    def start(self):
        if not self.ok:
            return
        self.stop_flag = False
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        if not self.ok:
            return None
        self.stop_flag = True
        self.thread.join()
        if not self.samples:
            return None
        reasons = sorted({name for _, bits in self.samples for b, name in self.REASONS.items() if bits & b})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml"}


# ------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ workloads
def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "conv_bn_activation_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name, src_files):
    """DRAM bytes per launch recorded in a profiles/ summary, if the kernel source is unchanged since."""
    p = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(p):
        return None
    text = open(p).read()
    m_hash = re.search(r"source-hash:\s*([0-9a-f]{16})", text)
    m_tr = re.search(r"traffic-bytes-per-launch:\s*([0-9]+)", text)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash(src_files):
        return None
    return int(m_tr.group(1))


class DepthwiseWorkload:
    name = "depthwise3x3_bn_relu"

    def __init__(self, torch, device, batch=64):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import ConvBnAct
        self.torch = torch
        self.x_host, w, bn = synthetic.depthwise_layer(N=batch)
        self.w, self.bn = w, bn
        self.batch = batch
        self.x = torch.from_numpy(self.x_host).to(device)
        self.l1 = ConvBnAct(w, bn, 1, 1, cb.ACT_RELU, groups=384, device=device)
        self.l2 = ConvBnAct(w, bn, 2, 1, cb.ACT_RELU, groups=384, device=device)
        self.y1 = torch.empty(batch, 56, 56, 384, device=device)
        self.y2 = torch.empty(batch, 28, 28, 384, device=device)
        wl = workloads.depthwise_workload(N=batch)
        self.work = {"s1": wl["s1"], "s2": wl["s2"]}
        self.step_bytes = wl["s1"].bytes + wl["s2"].bytes
        self.launches = ["s1", "s2"]
        self.config = {"workload": "depthwise 3x3 + BN + ReLU, NHWC fp32, N=64 C=384 56x56, stride 1 and 2",
                       "batch": batch, "l2": "inputs_larger_than_l2 (308 MB input, 129 MB L2)"}
        self.unit, self.per_image = "GB/s", True

    def run(self, stream, events=None):
        if events:
            events[0].record(stream)
        self.l1(self.x, self.y1, stream=stream)
        if events:
            events[1].record(stream)
        self.l2(self.x, self.y2, stream=stream)
        if events:
            events[2].record(stream)

    def e2e_setup(self):
        t = self.torch
        self.x_pin = t.from_numpy(self.x_host).pin_memory()
        self.y1_pin = t.empty(tuple(self.y1.shape), pin_memory=True)
        self.y2_pin = t.empty(tuple(self.y2.shape), pin_memory=True)
        return self.x_pin.numel() * 4, (self.y1_pin.numel() + self.y2_pin.numel()) * 4

    def e2e_step(self, stream):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.run(stream)
        self.y1_pin.copy_(self.y1, non_blocking=True)
        self.y2_pin.copy_(self.y2, non_blocking=True)

    def roofline(self, launch_ms, peaks, gpu_launch_name="s1"):
        ms = launch_ms[gpu_launch_name]
        achieved = self.work[gpu_launch_name].bytes / (ms * 1e-3) / 1e9
        traffic = profiled_traffic("dw_tma_kernel_depthwise_64x56x56x384.md", ["dw_conv.cu", "ptx.cuh", "epilogue.cuh"])
        return {"bound": "hbm", "kernel": "cb::dw_tma_kernel<1> (stride 1 launch)", "achieved": round(achieved, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes": self.work[gpu_launch_name].bytes,
                "peak_source": f"{peaks['source']} hbm_gbs (copy-kernel burst)"}

    def cpu_sample(self, n_images):
        import oracle
        x = self.x_host[:n_images]
        t0 = time.perf_counter()
        oracle.conv_bn_act(x, self.w, self.bn, stride=1, pad=1, groups=384, act=oracle.ACT_RELU)
        oracle.conv_bn_act(x, self.w, self.bn, stride=2, pad=1, groups=384, act=oracle.ACT_RELU)
        dt = time.perf_counter() - t0
        return dt, self.step_bytes * n_images / self.batch


def make_workload(name, torch, device):
    if name == "depthwise":
        return DepthwiseWorkload(torch, device)
    from bench_workloads import make  # the other measurement workloads
    return make(name, torch, device)


# ------------------------------------------------------------ arms
def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from conv_bn_activation_gb300 import _build, binding
    _build.build_library()
    binding.load()
    peaks = load_peaks()

    wl = make_workload(args.workload, torch, device)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        wl.run(stream)
    torch.cuda.synchronize()
    if binding.get_device_error() != binding.OK:
        raise RuntimeError("device error during warm-up")

    nl = len(wl.launches)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(args.steps)]
    sampler = ClockSampler(torch, local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    t_host0 = time.perf_counter()
    for k in range(args.steps):
        wl.run(stream, events[k])
    torch.cuda.synchronize()
    t_host = time.perf_counter() - t_host0
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [events[k][0].elapsed_time(events[k][nl]) for k in range(args.steps)]
    total_ms = events[0][0].elapsed_time(events[-1][nl])
    launch_ms = {name: statistics.mean(events[k][i].elapsed_time(events[k][i + 1]) for k in range(args.steps))
                 for i, name in enumerate(wl.launches)}
    if binding.get_device_error() != binding.OK:
        raise RuntimeError("device error during the timed steps")

    # e2e: host buffers, copies inside the timed region
    h2d, d2h = wl.e2e_setup()
    for _ in range(max(1, args.warmup // 2)):
        wl.e2e_step(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 10))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        wl.e2e_step(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps

    units = wl.step_bytes * args.steps
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms, e2e_ms = float(t[0]), float(t[1])
        u = torch.tensor([float(units)], dtype=torch.float64, device=device)
        dist.all_reduce(u)
        units = float(u[0])
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    value = units / (total_ms * 1e-3) / 1e9
    e2e_value = wl.step_bytes * world / (e2e_ms * 1e-3) / 1e9
    line = {
        "metric": "fused conv+BN+act: achieved GB/s or TFLOP/s vs roofline; images/sec",
        "value": round(value, 2), "unit": wl.unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(wl.config, parallelism=f"replicas x{world} (independent images, no collective)"),
        "images_per_s": round(wl.batch * world * args.steps / (total_ms * 1e-3), 1),
        "step_ms": {"median": round(statistics.median(step_ms), 4), "min": round(min(step_ms), 4),
                    "max": round(max(step_ms), 4)},
        "launch_ms": {k: round(v, 4) for k, v in launch_ms.items()},
        "roofline": wl.roofline(launch_ms, peaks),
        "e2e": {"value": round(e2e_value, 3), "unit": wl.unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 3)},
        "gpu_launches": nl * args.steps,
        "clocks": clocks,
        "host_wall_s": round(t_host, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(wl, target_s=12.0):
    import oracle
    oracle.build()
    dt1, _ = wl.cpu_sample(1)
    n = int(max(1, min(wl.batch, target_s / max(dt1, 1e-3))))
    dt, nbytes = wl.cpu_sample(n)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": wl.unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} of {wl.batch} images of the same workload (fp64 oracle, OpenMP)",
            "seconds": round(dt, 2)}


def run_reference(args):
    """The oracle as the reference arm, on the host cores, rank 0 only."""
    world, rank, local = dist_setup()
    if rank != 0:
        return
    import oracle
    oracle.build()

    wl = ReferenceDepthwise()
    for _ in range(args.warmup):
        wl.step()
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += wl.step()
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference",
        "metric": "fused conv+BN+act: achieved GB/s or TFLOP/s vs roofline; images/sec",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "depthwise 3x3 + BN + ReLU, NHWC fp32, N=64 C=384 56x56, stride 1 and 2",
                   "batch": 64, "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{wl.n} image(s) of the 64-image batch per step, stride 1 and 2"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


class ReferenceDepthwise:
    def __init__(self, n=1):
        from conv_bn_activation_gb300 import synthetic, workloads
        self.x, self.w, self.bn = synthetic.depthwise_layer()
        self.n = n
        wl = workloads.depthwise_workload()
        self.bytes = (wl["s1"].bytes + wl["s2"].bytes) * n // 64

    def step(self):
        import oracle
        x = self.x[:self.n]
        oracle.conv_bn_act(x, self.w, self.bn, stride=1, pad=1, groups=384, act=oracle.ACT_RELU)
        oracle.conv_bn_act(x, self.w, self.bn, stride=2, pad=1, groups=384, act=oracle.ACT_RELU)
        return self.bytes


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="depthwise",
                    choices=["depthwise", "dense", "mnist", "yolo", "preprocess"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
