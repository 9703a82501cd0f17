"""Benchmark of the fused conv + BN + activation hot path on GB300.

Default workload (N=1): the YOLO-style 20-conv chain, NHWC fp32, x =
[32, 640, 640, 3] ~ U[0,1], five stages of conv3x3 s2 -> 1x1 -> 3x3 -> 1x1
over the channel concat with a post-activation residual, every conv + BN +
SiLU.  ``value`` is images per second over the timed steps, whole job (all
ranks).  A step is R passes of the chain over the batch, R chosen so that
the timed region lasts at least --min-timed-s (the pass count is in
``config``); the R passes of a step are one CUDA graph.

The same line carries, under ``configs``, the other configurations measured
in the same run, each with its value, roofline and CPU baseline:
  mnist       the DepthwiseMNIST forward at batch 64 (images/s)
  depthwise   the depthwise 3x3 + BN + ReLU layer [64,56,56,384], stride 1 and 2 (GB/s)
  dense       the dense 3x3 + BN + SiLU sweep at batch 16 and 1 (TFLOP/s, tensor cores)
  yolo        the chain at batch 1
  preprocess  fused u8 preprocess -> stem conv at batch 32 (GB/s on the page's ledger)
Each of these (and the bf16 storage and pointwise variants) can also be run
alone with ``--workload``.

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

METRIC = "fused conv+BN+act: achieved GB/s or TFLOP/s vs roofline; images/sec"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
AUTOTUNE = True  # measure the tile plans of tensor-core layers at setup (cb_autotune_conv)
TF32_OVER_BF16 = 1.1 / 2.25  # nominal dense TF32 / BF16 tensor rates
# kind::tf32 MMAs (M = 128, N = 256, K = 8) issued back to back on all 152 SMs of a GB300 at
# 2070 MHz, 128 cycles each: the rate the TF32 tensor pipe sustains, reported beside the peak
# scaled from the bf16 measurement
TF32_ISSUE_LOOP_TFLOPS = 1207.0
UNIT_SCALE = {"GB/s": 1e9, "TFLOP/s": 1e12, "images/s": 1.0}


FP32_LANES_PER_SM = 128  # fp32 FMA lanes per SM (4 partitions x 32)
MAX_SM_MHZ = 2070        # maximum SM clock of this part


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def tf32_peak(peaks, sustained=False):
    return (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]) * TF32_OVER_BF16


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


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_over_ranks(torch, total_ms, e2e_ms, units, e2e_units, device):
    """Whole-job figures over the ranks of the default process group (any backend): the time is
    the slowest rank's, the units are summed (each rank runs its own batch: weak scaling)."""
    import torch.distributed as dist
    t = torch.tensor([total_ms, e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor([float(units), float(e2e_units)], dtype=torch.float64, device=device)
    dist.all_reduce(u)
    return float(t[0]), float(t[1]), float(u[0]), float(u[1])


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


# ------------------------------------------------------------ workloads
PATH_KERNELS = {1: ("cb::direct_tile_kernel / direct_conv_kernel", "hbm"), 2: ("cb::dw_tma_kernel", "hbm"),
                3: ("cb::igemm_tf32_kernel", "tensor"), 4: ("cb::igemm_halo_kernel (pixel-major)", "tensor"),
                5: ("cb::igemm_halo_kernel (channel-major)", "tensor"), 6: ("cb::pw_small_kernel", "hbm"),
                7: ("cb::stem_tc_kernel / stem_kernel", "hbm")}


def kernel_of(binding, x, y, k, stride, pad, x_layout=0):
    """(kernel name, roofline bound) of the path the library takes for this layer."""
    return PATH_KERNELS.get(binding.conv_path(x, y, k, stride, pad, x_layout=x_layout), ("?", "hbm"))


class Launch:
    def __init__(self, name, fn, work, kernel, bound):
        self.name, self.fn, self.work, self.kernel, self.bound = name, fn, work, kernel, bound


class Workload:
    """A step = the listed launches, in order, on one stream."""
    unit = "GB/s"
    tc_dtype = "tf32"       # operand type of the tensor-core launches: the roofline takes that type's peak
    capture = True          # time the K steps as one CUDA graph (no host gaps between launches)
    profile = None          # (profiles/ file, kernel source files) for the roofline's traffic figure
    profiles = {}           # the same per launch name, for workloads whose dominant launch varies
    dominant = None         # launch name whose roofline is reported

    def run(self, stream, events=None):
        for i, L in enumerate(self.launches):
            if events:
                events[i].record(stream)
            L.fn(stream)
        if events:
            events[len(self.launches)].record(stream)

    def time_launches(self, torch, stream, device, reps=20, eager=False):
        """ms per launch: `reps` back-to-back launches of each step entry (one CUDA
        graph unless eager), timed with events around them."""
        out = {}
        for L in self.launches:
            g = None
            if self.capture and not eager:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    cap = torch.cuda.current_stream(device)
                    for _ in range(reps):
                        L.fn(cap)
                g.replay()
            else:
                for _ in range(2):
                    L.fn(stream)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            if g is not None:
                g.replay()
            else:
                for _ in range(reps):
                    L.fn(stream)
            e1.record(stream)
            torch.cuda.synchronize()
            out[L.name] = e0.elapsed_time(e1) / reps
            del g
        return out

    def step_units(self):
        if self.unit == "GB/s":
            return sum(L.work.bytes for L in self.launches)
        if self.unit == "TFLOP/s":
            return sum(L.work.flops for L in self.launches)
        return self.batch

    def launch_roofline(self, L, ms, peaks):
        if L.bound == "tensor":
            achieved = L.work.flops / (ms * 1e-3) / 1e12
            peak = peaks["bf16_tflops"] if self.tc_dtype == "bf16" else tf32_peak(peaks)
            bw_roof = L.work.bytes / (ms * 1e-3) / 1e9
            r = {"bound": "tensor", "achieved": round(achieved, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                 "frac": round(achieved / peak, 4),
                 "frac_of_min_roof": round(achieved / min(peak, L.work.intensity * peaks["hbm_gbs"] / 1e3), 4),
                 "hbm_gbs": round(bw_roof, 1), "intensity": round(L.work.intensity, 2)}
            if self.tc_dtype != "bf16":
                r["frac_of_tf32_issue_loop"] = round(achieved / TF32_ISSUE_LOOP_TFLOPS, 4)
            return r
        if L.bound == "alu":  # fp32 FMAs on the CUDA cores: against the derived FMA peak
            achieved = L.work.flops / (ms * 1e-3) / 1e12
            return {"bound": "alu", "achieved": round(achieved, 2), "peak": round(peaks["fp32_fma_tflops"], 1),
                    "unit": "TFLOP/s", "frac": round(achieved / peaks["fp32_fma_tflops"], 4),
                    "hbm_gbs": round(L.work.bytes / (ms * 1e-3) / 1e9, 1),
                    "hbm_frac": round(L.work.bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        achieved = L.work.bytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4)}

    def roofline(self, launch_ms, peaks):
        L = next(l for l in self.launches if l.name == self.dominant) if self.dominant else \
            max(self.launches, key=lambda l: launch_ms[l.name])
        r = self.launch_roofline(L, launch_ms[L.name], peaks)
        r["kernel"] = f"{L.kernel} ({L.name})"
        r["algorithmic_bytes" if r["bound"] == "hbm" else "algorithmic_flops"] = \
            L.work.bytes if r["bound"] == "hbm" else L.work.flops
        if r["bound"] == "alu":
            r["algorithmic_bytes"] = L.work.bytes
        prof = self.profiles.get(L.name, self.profile)
        r["traffic"] = profiled_traffic(*prof) if prof else None
        if r["bound"] == "hbm":
            r["peak_source"] = f"{peaks['source']} hbm_gbs (copy-kernel burst)"
        elif r["bound"] == "alu":
            r["peak_source"] = ("derived: SMs x 128 fp32 lanes x 2 FLOP per FMA x 2070 MHz maximum SM clock "
                                f"({peaks['sms']} SMs)")
        elif self.tc_dtype == "bf16":
            r["peak_source"] = f"{peaks['source']} bf16_tflops (cuBLAS bf16 burst)"
        else:
            r["peak_source"] = f"{peaks['source']} bf16_tflops x 1.1/2.25 (nominal TF32/BF16 ratio)"
        return r

    def per_launch(self, launch_ms, peaks):
        out = {}
        for L in self.launches:
            r = self.launch_roofline(L, launch_ms[L.name], peaks)
            out[L.name] = {"us": round(launch_ms[L.name] * 1e3, 2), "kernel": L.kernel, "bound": r["bound"],
                           "achieved": r["achieved"], "unit": r["unit"], "frac": r["frac"]}
            if "frac_of_min_roof" in r:
                out[L.name]["frac_of_min_roof"] = r["frac_of_min_roof"]
        return out


def _t(torch, a, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DepthwiseWorkload(Workload):
    unit = "GB/s"
    dominant = "s1"
    profile = ("dw_tma_kernel_depthwise_64x56x56x384.md", ["dw_conv.cu", "ptx.cuh", "epilogue.cuh", "launch_util.h"])

    def __init__(self, torch, device, batch=64):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import ConvBnAct
        self.torch, self.batch = torch, batch
        self.x_host, self.w, self.bn = synthetic.depthwise_layer(N=batch)
        self.x = _t(torch, self.x_host, device)
        self.l1 = ConvBnAct(self.w, self.bn, 1, 1, cb.ACT_RELU, groups=384, device=device)
        self.l2 = ConvBnAct(self.w, self.bn, 2, 1, cb.ACT_RELU, groups=384, device=device)
        self.y1 = torch.empty(batch, 56, 56, 384, device=device)
        self.y2 = torch.empty(batch, 28, 28, 384, device=device)
        wl = workloads.depthwise_workload(N=batch)
        self.launches = [
            Launch("s1", lambda s: self.l1(self.x, self.y1, stream=s), wl["s1"], "cb::dw_tma_kernel<1,RELU,NONE>", "hbm"),
            Launch("s2", lambda s: self.l2(self.x, self.y2, stream=s), wl["s2"], "cb::dw_tma_kernel<2,RELU,NONE>", "hbm"),
        ]
        self.config = {"workload": "depthwise 3x3 + BN + ReLU, NHWC fp32, N=64 C=384 56x56, stride 1 and 2",
                       "batch": batch, "l2": "inputs_larger_than_l2 (308 MB input, 129 MB L2)"}

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

    def cpu_sample(self, n):
        import oracle
        x = self.x_host[:n]
        t0 = time.perf_counter()
        oracle.conv_bn_act(x, self.w, self.bn, stride=1, pad=1, groups=384, act=oracle.ACT_RELU)
        oracle.conv_bn_act(x, self.w, self.bn, stride=2, pad=1, groups=384, act=oracle.ACT_RELU)
        return time.perf_counter() - t0, self.step_units() * n / self.batch, f"{n} of {self.batch} images"


class DenseWorkload(Workload):
    unit = "TFLOP/s"
    dominant = "256-256@20_s1"
    bf16 = False

    def __init__(self, torch, device, batch=16):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import ConvBnAct
        self.torch, self.batch = torch, batch
        self.layers = []
        self.launches = []
        dt = torch.bfloat16 if self.bf16 else torch.float32
        eb = 2 if self.bf16 else 4
        # bf16 storage: the tensor-core layers (the 3-channel stem has no bf16 kernel)
        sweep = synthetic.DENSE_SWEEP[1:] if self.bf16 else synthetic.DENSE_SWEEP
        for (ci, co, H, s) in sweep:
            x, w, bn = synthetic.dense_layer(ci, co, H, N=batch, k=3)
            L = ConvBnAct(w, bn, s, 1, cb.ACT_SILU, device=device, dtype=dt)
            OH, OW = L.out_hw(H, H)
            xt = torch.from_numpy(x).to(dt)
            rec = {"x_host": xt.float().numpy(), "x_pin_src": xt, "w": w, "bn": bn, "s": s, "x": xt.to(device),
                   "y": torch.empty(batch, OH, OW, co, dtype=dt, device=device), "L": L}
            if AUTOTUNE:
                L.autotune(rec["x"], rec["y"])
            self.layers.append(rec)
            name = f"{ci}-{co}@{H}_s{s}"
            kname, bound = kernel_of(cb, rec["x"], rec["y"], 3, s, 1)
            tc = L.tc_weights
            self.launches.append(Launch(name, (lambda r: lambda st: r["L"](r["x"], r["y"], stream=st))(rec),
                                        workloads.conv_layer(batch, H, H, ci, co, 3, s, 1, act_bytes=eb,
                                                             w_bytes=eb if tc else 4), kname, bound))
        storage = ("NHWC bf16 storage, bf16 tensor-core operands (fp32 accumulate), the 7 tensor-core layers"
                   if self.bf16 else "NHWC fp32 storage, TF32 tensor cores")
        self.config = {"workload": f"dense 3x3 + BN + SiLU sweep, {storage}, batch {batch}",
                       "batch": batch, "l2": "warm (per-layer working sets 15-180 MB; steps run back to back)",
                       "autotune": AUTOTUNE}

    def e2e_setup(self):
        t = self.torch
        h2d = d2h = 0
        for r in self.layers:
            r["x_pin"] = r["x_pin_src"].pin_memory()
            r["y_pin"] = t.empty(tuple(r["y"].shape), dtype=r["y"].dtype, pin_memory=True)
            h2d += r["x_pin"].numel() * r["x_pin"].element_size()
            d2h += r["y_pin"].numel() * r["y_pin"].element_size()
        return h2d, d2h

    def e2e_step(self, stream):
        for r in self.layers:
            r["x"].copy_(r["x_pin"], non_blocking=True)
        self.run(stream)
        for r in self.layers:
            r["y_pin"].copy_(r["y"], non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        t0 = time.perf_counter()
        for r in self.layers:
            oracle.conv_bn_act(r["x_host"][:n], r["w"], r["bn"], stride=r["s"], pad=1, act=oracle.ACT_SILU)
        return time.perf_counter() - t0, self.step_units() * n / self.batch, f"{n} of {self.batch} images per layer"


class DenseBf16Workload(DenseWorkload):
    """The tensor-core layers of the dense sweep with bf16 storage and bf16 MMA operands."""
    bf16 = True
    tc_dtype = "bf16"


class MnistWorkload(Workload):
    """The whole DepthwiseMNIST forward, replayed as one CUDA graph per step."""
    unit = "images/s"
    capture = False  # already one graph launch per step

    def __init__(self, torch, device, batch=64):
        from conv_bn_activation_gb300 import synthetic, workloads
        from conv_bn_activation_gb300.nets import MnistNet
        self.torch, self.batch = torch, batch
        self.params = synthetic.mnist_params()
        self.x_host = synthetic.mnist_input(batch)
        self.x = _t(torch, self.x_host, device)
        self.net = MnistNet(self.params, batch, device=device)
        self.net.forward(self.x)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(device)
        side.wait_stream(torch.cuda.current_stream(device))
        with torch.cuda.stream(side):
            self.net.forward(self.x)
        torch.cuda.current_stream(device).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.net.forward(self.x)
        total = workloads.total(workloads.mnist_layers(N=batch))
        self.launches = [Launch("forward_graph", lambda s: self.graph.replay(), total,
                                "CUDA graph: stem + 4 blocks + pool/fc (13 kernels)", "hbm")]
        self.kernels_per_step = 13
        self.config = {"workload": "DepthwiseMNIST forward (stem, 4 depthwise-separable blocks, avgpool+fc), fp32",
                       "batch": batch, "l2": "warm (whole net ~40 MB fits in L2; graph replay back to back)"}

    def e2e_setup(self):
        self.x_pin = self.torch.from_numpy(self.x_host).pin_memory()
        self.out_pin = self.torch.empty(self.batch, 10, pin_memory=True)
        return self.x_pin.numel() * 4, self.out_pin.numel() * 4

    def e2e_step(self, stream):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.run(stream)
        self.out_pin.copy_(self.net.logits, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        t0 = time.perf_counter()
        oracle.mnist_model(self.x_host[:n], self.params)
        return time.perf_counter() - t0, n, f"{n} of {self.batch} images"


class YoloWorkload(Workload):
    unit = "images/s"
    # ncu summaries (DRAM traffic of one launch at batch 32) of the launches that can be the longest
    profiles = {
        "s0.down": ("stem_tc_kernel_yolo_s0_down_b32.md",
                    ["stem_tc.cu", "epilogue.cuh", "ptx.cuh", "tc_store.cuh", "launch_util.h", "internal.h"]),
        "s0.body": ("stage_body_kernel_yolo_s0_body_b32.md",
                    ["stage_body.cu", "epilogue.cuh", "ptx.cuh", "launch_util.h", "internal.h"]),
        "s1.body": ("stage_body_tc_kernel_yolo_s1_body_b32.md",
                    ["stage_body_tc.cu", "epilogue.cuh", "ptx.cuh", "tc_store.cuh", "launch_util.h", "internal.h"]),
        "s0.cv2": ("conv3x3_c8_kernel_yolo_s0_cv2_b32.md",
                   ["conv3x3_c8.cu", "epilogue.cuh", "ptx.cuh", "launch_util.h", "internal.h"]),
        "s0.cv3": ("pw_small_kernel_yolo_s0_cv3_b32.md",
                   ["pointwise.cu", "epilogue.cuh", "ptx.cuh", "launch_util.h", "internal.h"]),
    }

    bf16 = False

    def __init__(self, torch, device, batch=32):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import YoloChain
        self.torch, self.batch = torch, batch
        self.stages = synthetic.yolo_params()
        dt = torch.bfloat16 if self.bf16 else torch.float32
        self.x_src = torch.from_numpy(synthetic.yolo_input(batch)).to(dt)
        self.x_host = self.x_src.float().numpy()  # the values the chain reads, for the oracle
        self.x = self.x_src.to(device)
        self.chain = YoloChain(self.stages, batch, device=device, dtype=dt)
        if AUTOTUNE:
            self.chain.forward(self.x, tune=True)
        eb = 2 if self.bf16 else 4
        works = dict(workloads.yolo_layers(
            N=batch, act_bytes=eb,
            tc_w_bytes=lambda ci, co, k, s: eb if cb.layer_uses_tensor_cores(ci, co, k, s) else 4))
        self.launches = []
        prev = lambda: self.x
        for i, (L, B) in enumerate(zip(self.chain.layers, self.chain.bufs)):
            half = B["half"]
            a, b = B["cat"][..., :half], B["cat"][..., half:]
            x_in = prev
            steps = [
                ("down", (lambda L=L, B=B, x_in=x_in: lambda s: L["down"](x_in(), B["x1"], stream=s))()),
                ("cv1", (lambda L=L, B=B, a=a: lambda s: L["cv1"](B["x1"], a, stream=s))()),
                ("cv2", (lambda L=L, a=a, b=b: lambda s: L["cv2"](a, b, stream=s))()),
                ("cv3", (lambda L=L, B=B: lambda s: L["cv3"](B["cat"], B["out"], residual=B["x1"],
                                                             res_mode=cb.RES_POST_ACT, stream=s))()),
            ]
            views = {"down": (x_in(), B["x1"]), "cv1": (B["x1"], a), "cv2": (a, b), "cv3": (B["cat"], B["out"])}
            if self.chain.fused[i]:  # the stage body as one kernel (cb_stage_body)
                x1 = B["x1"]
                steps = steps[:1] + [("body", (lambda i=i: lambda s: self.chain.body(i, stream=s))())]
                works[f"s{i}.body"] = workloads.stage_body(batch, x1.shape[1], x1.shape[2], x1.shape[3], eb)
            for nm, fn in steps:
                if nm == "body":  # 16 channels: fp32 FMAs on the CUDA cores; 32: the tensor cores
                    kname, bound = (("cb::stage_body_kernel", "alu") if B["x1"].shape[3] == 16 else
                                    ("cb::stage_body_tc_kernel", "tensor"))
                else:
                    xv, yv = views[nm]
                    kname, bound = kernel_of(cb, xv, yv, L[nm].k, L[nm].stride, L[nm].pad)
                self.launches.append(Launch(f"s{i}.{nm}", fn, works[f"s{i}.{nm}"], kname, bound))
            prev = (lambda B=B: lambda: B["out"])()
        storage = ("bf16 storage: every layer reads and writes bf16, tensor-core layers multiply bf16 "
                   "weights, fp32 accumulation" if self.bf16 else "fp32")
        self.config = {"workload": "YOLO-style 20-conv chain (5 stages, concat via channel views, post-act "
                                   "residual; the 16- and 32-channel stage bodies as one kernel each), "
                                   f"640x640x3, {storage}",
                       "batch": batch,
                       "l2": f"inputs_larger_than_l2 ({157 * eb // 4} MB input, {1.2 * eb / 4:.1f} GB of "
                             "activations per step)",
                       "autotune": AUTOTUNE}

    def e2e_setup(self):
        t = self.torch
        self.x_pin = self.x_src.pin_memory()
        out = self.chain.bufs[-1]["out"]
        self.out_pin = t.empty(tuple(out.shape), dtype=out.dtype, pin_memory=True)
        # a second device input buffer and a copy stream: step i + 1's input
        # crosses the link while step i computes; the outputs leave on a third
        # stream, so that they do not queue behind the next input (the link
        # carries both directions at once)
        self.x_bufs = [self.x, t.empty_like(self.x)]
        self.copy_stream = t.cuda.Stream(self.x.device)
        self.d2h_stream = t.cuda.Stream(self.x.device)
        return (self.x_pin.numel() * self.x_pin.element_size(),
                self.out_pin.numel() * self.out_pin.element_size())

    def e2e_step(self, stream):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.run(stream)
        self.out_pin.copy_(self.chain.bufs[-1]["out"], non_blocking=True)

    def e2e_pipelined(self, stream, steps):
        """`steps` steps with host buffers, each: the H2D copy of its input (pinned), the chain, the
        D2H copy of its output.  The copies run on two more streams: the input into two alternating
        device buffers one step ahead of the chain, the output after the chain is done with it
        (the next step's last layer, which rewrites that buffer, waits for the copy)."""
        t = self.torch
        copy, out_s = self.copy_stream, self.d2h_stream
        h2d = [t.cuda.Event(), t.cuda.Event()]
        free = [t.cuda.Event(), t.cuda.Event()]
        done, d2h = t.cuda.Event(), t.cuda.Event()
        copy.wait_stream(stream)
        out_s.wait_stream(stream)

        def issue_h2d(i):
            b = i & 1
            with t.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(free[b])      # the chain of step i - 2 is done with buffer b
                self.x_bufs[b].copy_(self.x_pin, non_blocking=True)
                h2d[b].record(copy)

        issue_h2d(0)
        last = len(self.launches) - 1
        for i in range(steps):
            if i + 1 < steps:
                issue_h2d(i + 1)
            b = i & 1
            stream.wait_event(h2d[b])
            self.x = self.x_bufs[b]
            for k, L in enumerate(self.launches):
                if k == last and i > 0:
                    stream.wait_event(d2h)            # step i - 1's output has been copied out
                L.fn(stream)
            free[b].record(stream)
            done.record(stream)
            with t.cuda.stream(out_s):
                out_s.wait_event(done)
                self.out_pin.copy_(self.chain.bufs[-1]["out"], non_blocking=True)
                d2h.record(out_s)
        stream.wait_stream(copy)
        stream.wait_stream(out_s)
        self.x = self.x_bufs[0]

    def cpu_sample(self, n):
        import oracle
        t0 = time.perf_counter()
        h = self.x_host[:n]
        for st in self.stages:
            h = oracle.yolo_stage(h, st).astype(np.float32)
        return time.perf_counter() - t0, n, f"{n} of {self.batch} images"


class YoloBf16Workload(YoloWorkload):
    """The YOLO-style chain with bf16 storage."""
    bf16 = True
    tc_dtype = "bf16"
    # the fp32 chain's summaries are of other kernel instances: only the bf16 ones apply
    profiles = {
        "s1.body": ("stage_body_tc_kernel_yolo_bf16_s1_body_b32.md",
                    ["stage_body_tc.cu", "epilogue.cuh", "ptx.cuh", "tc_store.cuh", "launch_util.h", "internal.h"]),
    }


class PreprocessWorkload(Workload):
    """u8 frames -> resize + /255 -> stem conv, as one kernel (the preprocess fused into the stem's
    input staging).  The preprocess kernel alone (its own byte ledger), the two-kernel path
    (preprocess to memory, then the stem) and the three-pass path are timed beside it."""
    unit = "GB/s"
    dominant = "preprocess_stem"
    profile = ("stem_kernel_preprocess_32x1280x720.md",
               ["stem.cu", "resample.cuh", "epilogue.cuh", "ptx.cuh", "launch_util.h", "internal.h"])

    def __init__(self, torch, device, batch=32):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import PreprocessStem
        self.torch, self.batch = torch, batch
        self.frames_host = synthetic.preprocess_frames(N=batch)
        self.frames = _t(torch, self.frames_host, device)
        self.sw, self.sbn = synthetic.stem_params()
        self.net = PreprocessStem(self.sw, self.sbn, batch, device=device)
        self.net.tmp_u8 = torch.empty(batch, 480, 640, 3, dtype=torch.uint8, device=device)
        self.net.tmp_f32 = torch.empty(batch, 480, 640, 3, device=device)
        work = workloads.preprocess_stem_fused(batch, 720, 1280, 480, 640)
        self.launches = [
            Launch("preprocess_stem", lambda s: self.net.forward(self.frames, stream=s), work,
                   "cb::stem_kernel (u8 frames: preprocess in the input staging)", "hbm"),
        ]
        self.pre = workloads.preprocess_fused(batch, 720, 1280, 480, 640)
        self.stem = workloads.conv_layer(batch, 480, 640, 3, 16, 3, 2, 1)
        self.three_pass = workloads.preprocess_unfused(batch, 720, 1280, 480, 640)
        self.config = {"workload": "u8 frames 1280x720 -> bilinear 640x480 -> /255 -> stem conv3x3 s2 3->16 + BN + "
                                   "SiLU (NHWC fp32 out), preprocess fused into the stem", "batch": batch,
                       "l2": "inputs_larger_than_l2 (88 MB frames + 157 MB stem out)",
                       "bytes_per_frame": work.bytes // batch}

    def extra(self, torch, stream, steps):
        """The preprocess kernel alone, the two-kernel path and the three-pass path, timed the same
        way (not part of the step)."""
        from conv_bn_activation_gb300 import binding as cb
        net = self.net

        def timed(fn):
            for _ in range(3):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / steps

        pre_ms = timed(lambda: cb.preprocess_u8(self.frames, net.planar, stream=stream))
        stem_ms = timed(lambda: net.stem(net.planar, net.out, stream=stream, x_layout=cb.LAYOUT_NCHW))
        two_ms = timed(lambda: net.forward(self.frames, stream=stream, fused=False))
        three_ms = timed(lambda: cb.preprocess_u8_three_pass(self.frames, net.tmp_u8, net.tmp_f32, net.planar,
                                                             stream=stream))
        hbm = load_peaks()["hbm_gbs"]
        pre_gbs = self.pre.bytes / (pre_ms * 1e-3) / 1e9
        ledger = workloads_ledger_ratio()
        return {"three_pass_over_fused_time": round(three_ms / pre_ms, 3),
                "page_predicted_ratio": round(ledger, 3),
                "ratio_note": "the page predicts the fused/unfused speed-up from its byte ledger "
                              "(15,667,200 / 6,451,200 B per frame); measured = three-pass time / fused time",
                "preprocess_kernel_us": round(pre_ms * 1e3, 2),
                "preprocess_kernel_gbs_on_its_ledger": round(pre_gbs, 1),
                "preprocess_kernel_frac": round(pre_gbs / hbm, 4),
                "stem_kernel_planar_us": round(stem_ms * 1e3, 2),
                "stem_kernel_planar_gbs": round(self.stem.bytes / (stem_ms * 1e-3) / 1e9, 1),
                "two_kernel_path_us": round(two_ms * 1e3, 2),
                "three_pass_us": round(three_ms * 1e3, 2),
                "three_pass_gbs_on_its_ledger": round(self.three_pass.bytes / (three_ms * 1e-3) / 1e9, 1),
                "ledger_bytes_per_frame": {"fused_preprocess": 6451200, "three_pass": 15667200,
                                           "preprocess_stem": self.launches[0].work.bytes // self.batch}}

    def e2e_setup(self):
        self.f_pin = self.torch.from_numpy(self.frames_host).pin_memory()
        self.out_pin = self.torch.empty(tuple(self.net.out.shape), pin_memory=True)
        return self.f_pin.numel(), self.out_pin.numel() * 4

    def e2e_step(self, stream):
        self.frames.copy_(self.f_pin, non_blocking=True)
        self.run(stream)
        self.out_pin.copy_(self.net.out, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        t0 = time.perf_counter()
        planar = oracle.preprocess_u8(self.frames_host[:n], 480, 640, oracle.PREC_F32)
        oracle.conv_bn_act(planar, self.sw, self.sbn, stride=2, pad=1, act=oracle.ACT_SILU, layout=oracle.NCHW)
        return time.perf_counter() - t0, self.step_units() * n / self.batch, f"{n} of {self.batch} frames"


def workloads_ledger_ratio():
    from conv_bn_activation_gb300 import workloads
    led = workloads.preprocess_ledger(720, 1280, 480, 640)
    return led["unfused"] / led["fused"]


class DepthwiseBf16Workload(DepthwiseWorkload):
    """The same layer with bf16 storage (x, y bf16; weights, scale, bias and arithmetic fp32)."""
    profile = ("dw_tma_kernel_depthwise_bf16_64x56x56x384.md",
               ["dw_conv.cu", "ptx.cuh", "epilogue.cuh", "launch_util.h"])

    def __init__(self, torch, device, batch=64):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import ConvBnAct
        self.torch, self.batch = torch, batch
        x, self.w, self.bn = synthetic.depthwise_layer(N=batch)
        xb = torch.from_numpy(x).to(torch.bfloat16)
        self.x_host = xb.float().numpy()          # the bf16 values, for the oracle
        self.x_host_bf16 = xb
        self.x = xb.to(device)
        self.l1 = ConvBnAct(self.w, self.bn, 1, 1, cb.ACT_RELU, groups=384, device=device)
        self.l2 = ConvBnAct(self.w, self.bn, 2, 1, cb.ACT_RELU, groups=384, device=device)
        self.y1 = torch.empty(batch, 56, 56, 384, dtype=torch.bfloat16, device=device)
        self.y2 = torch.empty(batch, 28, 28, 384, dtype=torch.bfloat16, device=device)
        wl = workloads.depthwise_workload(N=batch, act_bytes=2)
        self.launches = [
            Launch("s1", lambda s: self.l1(self.x, self.y1, stream=s), wl["s1"],
                   "cb::dw_tma_kernel<bf16,1,RELU,NONE>", "hbm"),
            Launch("s2", lambda s: self.l2(self.x, self.y2, stream=s), wl["s2"],
                   "cb::dw_tma_kernel<bf16,2,RELU,NONE>", "hbm"),
        ]
        self.config = {"workload": "depthwise 3x3 + BN + ReLU, NHWC bf16 storage (fp32 arithmetic), "
                                   "N=64 C=384 56x56, stride 1 and 2",
                       "batch": batch, "l2": "inputs_larger_than_l2 (154 MB input, 129 MB L2)"}

    def e2e_setup(self):
        t = self.torch
        self.x_pin = self.x_host_bf16.pin_memory()
        self.y1_pin = t.empty(tuple(self.y1.shape), dtype=t.bfloat16, pin_memory=True)
        self.y2_pin = t.empty(tuple(self.y2.shape), dtype=t.bfloat16, pin_memory=True)
        return self.x_pin.numel() * 2, (self.y1_pin.numel() + self.y2_pin.numel()) * 2


class PointwiseWorkload(Workload):
    """The two widest 1x1 layers of the YOLO-style chain at batch 32, 320x320: 16 -> 8 (+ SiLU) and
    16 -> 16 + SiLU with the post-activation residual; fp32 storage, or bf16 with bf16=True."""
    dominant = "cv3"
    bf16 = False

    def __init__(self, torch, device, batch=32):
        from conv_bn_activation_gb300 import binding as cb, synthetic, workloads
        from conv_bn_activation_gb300.nets import ConvBnAct
        self.torch, self.batch = torch, batch
        dt = torch.bfloat16 if self.bf16 else torch.float32
        eb = 2 if self.bf16 else 4
        H = 320
        x1, w1, bn1 = synthetic.dense_layer(16, 8, H, N=batch, k=1, seed=31)
        x3, w3, bn3 = synthetic.dense_layer(16, 16, H, N=batch, k=1, seed=33)
        r3 = synthetic.normal(synthetic.rng(35), (batch, H, H, 16))
        cast = lambda a: torch.from_numpy(a).to(dt)
        self.host = {"x1": cast(x1), "x3": cast(x3), "r3": cast(r3)}
        self.oracle_in = {k: v.float().numpy() for k, v in self.host.items()}
        self.w = {"cv1": (w1, bn1), "cv3": (w3, bn3)}
        self.x1, self.x3, self.r3 = (self.host[k].to(device) for k in ("x1", "x3", "r3"))
        self.l1 = ConvBnAct(w1, bn1, 1, 0, cb.ACT_SILU, device=device)
        self.l3 = ConvBnAct(w3, bn3, 1, 0, cb.ACT_SILU, device=device)
        self.y1 = torch.empty(batch, H, H, 8, dtype=dt, device=device)
        self.y3 = torch.empty(batch, H, H, 16, dtype=dt, device=device)
        self.launches = [
            Launch("cv1", lambda s: self.l1(self.x1, self.y1, stream=s),
                   workloads.conv_layer(batch, H, H, 16, 8, 1, 1, 0, act_bytes=eb),
                   f"cb::pw_small_kernel<16,8,{'bf16' if self.bf16 else 'f32'}>", "hbm"),
            Launch("cv3", lambda s: self.l3(self.x3, self.y3, residual=self.r3, res_mode=cb.RES_POST_ACT, stream=s),
                   workloads.conv_layer(batch, H, H, 16, 16, 1, 1, 0, residual=True, act_bytes=eb),
                   f"cb::pw_small_kernel<16,16,res,{'bf16' if self.bf16 else 'f32'}>", "hbm"),
        ]
        self.config = {"workload": f"pointwise 1x1 + BN + SiLU (YOLO stage-0 shapes 16->8 and 16->16 + residual), "
                                   f"NHWC {'bf16 storage (fp32 arithmetic)' if self.bf16 else 'fp32'}, N={batch} 320x320",
                       "batch": batch, "l2": "inputs_larger_than_l2"}

    def e2e_setup(self):
        t = self.torch
        self.pin = {k: v.pin_memory() for k, v in self.host.items()}
        self.y1_pin = t.empty(tuple(self.y1.shape), dtype=self.y1.dtype, pin_memory=True)
        self.y3_pin = t.empty(tuple(self.y3.shape), dtype=self.y3.dtype, pin_memory=True)
        eb = self.y1.element_size()
        return sum(v.numel() for v in self.pin.values()) * eb, (self.y1.numel() + self.y3.numel()) * eb

    def e2e_step(self, stream):
        self.x1.copy_(self.pin["x1"], non_blocking=True)
        self.x3.copy_(self.pin["x3"], non_blocking=True)
        self.r3.copy_(self.pin["r3"], non_blocking=True)
        self.run(stream)
        self.y1_pin.copy_(self.y1, non_blocking=True)
        self.y3_pin.copy_(self.y3, non_blocking=True)

    def cpu_sample(self, n):
        import oracle
        o = self.oracle_in
        t0 = time.perf_counter()
        oracle.conv_bn_act(o["x1"][:n], *self.w["cv1"], stride=1, pad=0, act=oracle.ACT_SILU)
        oracle.conv_bn_act(o["x3"][:n], *self.w["cv3"], stride=1, pad=0, act=oracle.ACT_SILU, residual=o["r3"][:n],
                           res_mode=oracle.RES_POST_ACT)
        return time.perf_counter() - t0, self.step_units() * n / self.batch, f"{n} of {self.batch} images"


class PointwiseBf16Workload(PointwiseWorkload):
    bf16 = True


WORKLOADS = {"depthwise": DepthwiseWorkload, "depthwise_bf16": DepthwiseBf16Workload, "pointwise": PointwiseWorkload,
             "pointwise_bf16": PointwiseBf16Workload, "dense": DenseWorkload, "dense_bf16": DenseBf16Workload,
             "mnist": MnistWorkload, "yolo": YoloWorkload, "yolo_bf16": YoloBf16Workload,
             "preprocess": PreprocessWorkload}


# ------------------------------------------------------------ arms
L2_FLUSH_BYTES = 320 << 20  # > 2x the 129 MB L2: written between cold-cache launch timings


def _percentile(sorted_vals, q):
    i = (len(sorted_vals) - 1) * q
    lo, hi = int(np.floor(i)), int(np.ceil(i))
    return sorted_vals[lo] + (sorted_vals[hi] - sorted_vals[lo]) * (i - lo)


def pass_graph(torch, wl, device, passes):
    """One CUDA graph of `passes` back-to-back passes of the workload (None for workloads that
    replay their own graph)."""
    if not wl.capture:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = torch.cuda.current_stream(device)
        for _ in range(passes):
            wl.run(cap)
    g.replay()
    torch.cuda.synchronize()
    return g


def replay(wl, graph, stream, passes):
    if graph is not None:
        graph.replay()
    else:
        for _ in range(passes):
            wl.run(stream)


def pass_stats(torch, wl, device, stream, reps=200):
    """Per-pass device time over `reps` single-pass replays with events between them: mean, P50,
    P95, P99 and the coefficient of variation (the metric list of "How I sped up convolutions")."""
    g = pass_graph(torch, wl, device, 1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    for _ in range(3):
        replay(wl, g, stream, 1)
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(reps):
        replay(wl, g, stream, 1)
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    ms = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(reps))
    mean = statistics.fmean(ms)
    return {"reps": reps, "mean_ms": round(mean, 4), "p50_ms": round(_percentile(ms, 0.50), 4),
            "p95_ms": round(_percentile(ms, 0.95), 4), "p99_ms": round(_percentile(ms, 0.99), 4),
            "cv": round(statistics.pstdev(ms) / mean, 4),
            "how": "single-pass graph replays, events between them (one event gap per pass)"}


def cold_launch_ms(torch, wl, device, stream, reps=7):
    """ms per launch with a cold L2: before each timed launch a buffer larger than twice the L2 is
    written (outside the events); median over reps."""
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    out = {}
    for L in wl.launches:
        ts = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            L.fn(stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        out[L.name] = statistics.median(ts)
    del flush
    return out


def short_kernel_name(mangled):
    """'cb::conv3x3_c8_kernel' from an Itanium-mangled name such as
    _ZN2cb12_GLOBAL__N_117conv3x3_c8_kernelILi2ELi0EEEvNS_10DirectArgsEii (anonymous namespaces
    skipped); the input itself when it is not of that form."""
    if not mangled or not mangled.startswith("_ZN"):
        return mangled
    parts, i = [], 3
    while i < len(mangled) and mangled[i].isdigit():
        j = i
        while j < len(mangled) and mangled[j].isdigit():
            j += 1
        k = int(mangled[i:j])
        name = mangled[j:j + k]
        i = j + k
        if not name.startswith("_GLOBAL__N"):
            parts.append(name)
    return "::".join(parts) if parts else mangled


def launch_occupancy(torch, wl, stream):
    """Per launch: grid, threads, shared memory and the CTAs per SM the occupancy calculator allows
    for the kernel the library launched (cb_last_launch)."""
    from conv_bn_activation_gb300 import binding
    out = {}
    if not wl.capture:
        return out
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    for L in wl.launches:
        L.fn(stream)
        info = binding.last_launch()
        info["kernel"] = short_kernel_name(info["kernel"])
        warps = info["blocks_per_sm"] * ((info["threads"] + 31) // 32)
        info["warps_per_sm"] = warps
        info["theoretical_occupancy"] = round(warps / 64.0, 3)   # 64 resident warps per SM
        info["waves"] = round(info["grid"] / max(1, info["blocks_per_sm"] * sms), 3)
        out[L.name] = info
    torch.cuda.synchronize()
    return out


def measure(torch, wl, device, stream, args, steps, warmup, min_timed_s, world, peaks, with_e2e, cpu_target_s):
    """The timed run of one workload: K steps of R passes each (R chosen so that the timed region
    lasts at least min_timed_s), with per-launch, cold-cache, statistics and occupancy figures."""
    from conv_bn_activation_gb300 import binding
    for _ in range(warmup):
        wl.run(stream)
    torch.cuda.synchronize()
    if binding.get_device_error() != binding.OK:
        raise RuntimeError("device error during warm-up")
    # passes per step: enough that the K timed steps last min_timed_s
    g1 = pass_graph(torch, wl, device, 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        replay(wl, g1, stream, 1)
    e1.record(stream)
    torch.cuda.synchronize()
    pass_ms = e0.elapsed_time(e1) / 5
    del g1
    passes = max(1, int(np.ceil(min_timed_s * 1e3 / (steps * max(pass_ms, 1e-3)))))
    # The R passes of a step are captured as one CUDA graph with no event
    # between launches: the library launches each kernel with programmatic
    # dependent launch, and an event between two kernels would serialise
    # them again.
    graph = pass_graph(torch, wl, device, passes)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch, device.index or 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    e_start.record(stream)
    for _ in range(steps):
        replay(wl, graph, stream, passes)
    e_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    total_ms = e_start.elapsed_time(e_end)
    del graph
    if binding.get_device_error() != binding.OK:
        raise RuntimeError("device error during the timed steps")
    # Per-kernel durations (the roofline's denominators): each launch of the
    # pass repeated back to back, events around the repetitions only; and
    # each launch alone after an L2 flush.
    launch_ms = wl.time_launches(torch, stream, device, reps=args.launch_reps, eager=args.eager)
    cold_ms = cold_launch_ms(torch, wl, device, stream) if wl.capture else {}
    stats = pass_stats(torch, wl, device, stream)
    occ = launch_occupancy(torch, wl, stream)
    if binding.get_device_error() != binding.OK:
        raise RuntimeError("device error while timing the launches")
    extra = wl.extra(torch, stream, 20) if hasattr(wl, "extra") else None

    # e2e: host buffers, copies inside the timed region, one pass per step
    h2d = d2h = 0
    e2e_ms = float("nan")
    if with_e2e:
        h2d, d2h = wl.e2e_setup()
        pipelined = hasattr(wl, "e2e_pipelined")
        for _ in range(3):
            wl.e2e_step(stream)
        if pipelined:
            wl.e2e_pipelined(stream, 3)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # the timed steps' count (at least 10, at most 50): a pipelined loop's first input copy,
        # which nothing overlaps, is then spread as it is in a serving loop of that length
        e2e_steps = max(10, min(steps, 50))
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        if pipelined:
            wl.e2e_pipelined(stream, e2e_steps)
        else:
            for _ in range(e2e_steps):
                wl.e2e_step(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1) / e2e_steps

    units = wl.step_units() * passes * steps
    e2e_units = wl.step_units()
    if world > 1:
        total_ms, e2e_ms, units, e2e_units = aggregate_over_ranks(torch, total_ms, e2e_ms, units, e2e_units, device)
    scale = UNIT_SCALE[wl.unit]
    value = units / (total_ms * 1e-3) / scale
    for L in wl.launches:  # label each launch with the kernel the library actually ran
        if L.name in occ and occ[L.name]["kernel"] not in ("", "?"):
            L.kernel = occ[L.name]["kernel"]
    per_launch = wl.per_launch(launch_ms, peaks)
    total_launch = sum(launch_ms.values())
    for name, rec in per_launch.items():
        rec["share"] = round(launch_ms[name] / total_launch, 4)
        if name in cold_ms:
            rec["us_cold_l2"] = round(cold_ms[name] * 1e3, 2)
        if name in occ:
            rec["occupancy"] = occ[name]
    by_kernel = {}
    for L in wl.launches:
        k = L.kernel.split(" (")[0]
        by_kernel.setdefault(k, [0, 0.0])
        by_kernel[k][0] += 1
        by_kernel[k][1] += launch_ms[L.name]
    out = {
        "value": round(value, 3), "unit": wl.unit, "steps": steps, "passes_per_step": passes,
        "ms_per_step": round(total_ms / steps, 4), "timed_region_s": round(total_ms / 1e3, 3),
        "config": dict(wl.config),
        "images_per_s": round(wl.batch * world * passes * steps / (total_ms * 1e-3), 1),
        "us_per_image": round(total_ms * 1e3 / (passes * steps) / wl.batch, 3),
        "step_stats": stats,
        "launches": per_launch,
        "kernel_shares": {k: {"launches": n, "us": round(t * 1e3, 2), "share": round(t / total_launch, 4)}
                          for k, (n, t) in sorted(by_kernel.items(), key=lambda kv: -kv[1][1])},
        "roofline": wl.roofline(launch_ms, peaks),
        "e2e": None if not with_e2e else {"value": round(e2e_units / (e2e_ms * 1e-3) / scale, 3), "unit": wl.unit,
                                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                          "ms_per_step": round(e2e_ms, 3),
                                          "step": "one pass with its host copies (pinned memory)" +
                                                  ("; the copies run on two more streams, one per "
                                                   "direction: the next step's input copy (two device input "
                                                   "buffers) and this step's output copy overlap the chains"
                                                   if hasattr(wl, "e2e_pipelined") else "")},
        "gpu_launches": getattr(wl, "kernels_per_step", len(wl.launches)) * passes * steps,
        "timing": {"steps": f"one CUDA graph of {passes} passes per step, replayed {steps} times, events around "
                            "all of them",
                   "launches": f"each launch repeated {args.launch_reps}x back to back "
                               f"({'eager' if args.eager or not wl.capture else 'one CUDA graph'}), "
                               "events around the repetitions; us_cold_l2: one launch after a 320 MB write, "
                               "median of 7"},
        "clocks": clocks,
    }
    if extra:
        out["comparison"] = extra
    if world == 1 and cpu_target_s > 0:
        out["cpu_baseline"] = cpu_baseline(wl, target_s=cpu_target_s, max_s=2.5 * cpu_target_s)
    return out


# The other configurations of the workload list, measured in the same run
# beside the headline one: (key, workload, batch).
EXTRA_CONFIGS = (("cfg0_mnist_b64", "mnist", 64), ("cfg1_depthwise_b64", "depthwise", 64),
                 ("cfg2_dense_b16", "dense", 16), ("cfg2_dense_b1", "dense", 1),
                 ("cfg3_yolo_b1", "yolo", 1), ("cfg4_preprocess_stem_b32", "preprocess", 32),
                 ("bf16_yolo_b32", "yolo_bf16", 32), ("bf16_dense_b16", "dense_bf16", 16),
                 ("bf16_depthwise_b64", "depthwise_bf16", 64),
                 ("bf16_pointwise_b32", "pointwise_bf16", 32))


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
    peaks["sms"] = torch.cuda.get_device_properties(device).multi_processor_count
    peaks["fp32_fma_tflops"] = peaks["sms"] * FP32_LANES_PER_SM * 2 * MAX_SM_MHZ * 1e6 / 1e12

    global AUTOTUNE
    AUTOTUNE = not args.no_autotune
    stream = torch.cuda.current_stream(device)
    wl = WORKLOADS[args.workload](torch, device, **({"batch": args.batch} if args.batch else {}))
    if args.profile_pass:
        # one pass inside an NVTX range, for profilers (ncu --nvtx --nvtx-include "profiled_pass/");
        # nothing is timed
        for _ in range(args.warmup):
            wl.run(stream)
        torch.cuda.synchronize()
        for L, info in zip(wl.launches, launch_occupancy(torch, wl, stream).values()):
            L.kernel = info["kernel"] or L.kernel  # the kernel the library launched
        torch.cuda.nvtx.range_push("profiled_pass")
        wl.run(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if binding.get_device_error() != binding.OK:
            raise RuntimeError("device error in the profiled pass")
        print(json.dumps({"profiled_pass": args.workload, "batch": wl.batch,
                          "launches": [[L.name, L.kernel] for L in wl.launches]}), flush=True)
        return
    main = measure(torch, wl, device, stream, args, args.steps, args.warmup, args.min_timed_s, world, peaks,
                   not args.no_e2e, 0 if args.no_cpu_baseline else 12.0)
    del wl
    extra = {}
    if args.workload == "yolo" and not args.batch and not args.no_extra_configs:
        for key, name, batch in EXTRA_CONFIGS:
            w = WORKLOADS[name](torch, device, batch=batch)
            r = measure(torch, w, device, stream, args, 10, 3, 0.3, world, peaks, False,
                        0 if args.no_cpu_baseline else 3.0)
            extra[key] = {k: r[k] for k in ("value", "unit", "config", "images_per_s", "us_per_image", "roofline",
                                            "step_stats", "launches", "kernel_shares", "cpu_baseline", "comparison",
                                            "passes_per_step", "ms_per_step")
                          if k in r}
            del w
            torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": main["value"], "unit": main["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(main["config"], passes_per_step=main["passes_per_step"],
                       parallelism=f"replicas x{world} (independent images, no collective)"),
    }
    line.update({k: v for k, v in main.items() if k not in ("value", "unit", "steps", "ms_per_step", "config")})
    if extra:
        line["configs"] = extra
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def cpu_baseline(wl, target_s=12.0, max_s=30.0):
    """The oracle as it stands, on the host cores, on a bounded sample of the workload: as many
    images of one step as fit in ~target_s, and when the whole step takes less, whole steps
    repeated until ~target_s (never past max_s)."""
    import oracle
    oracle.build()
    dt1, _, _ = wl.cpu_sample(1)
    n = int(max(1, min(wl.batch, target_s / max(dt1, 1e-3))))
    dt, units, what = wl.cpu_sample(n) if n > 1 else wl.cpu_sample(1)
    reps = 1
    while n == wl.batch and dt < target_s and dt * (reps + 1) / reps < max_s:
        d, u, _ = wl.cpu_sample(n)
        dt, units, reps = dt + d, units + u, reps + 1
    sample = f"{what} of the same workload" + (f", {reps} times" if reps > 1 else "") + " (fp64 oracle, OpenMP)"
    return {"value": round(units / dt / UNIT_SCALE[wl.unit], 6), "unit": wl.unit, "cores": oracle.num_threads(),
            "kind": "oracle", "sample": sample, "seconds": round(dt, 2)}


def run_reference(args):
    """The oracle as the reference arm, on the host cores, rank 0 only: the same workload, metric
    and unit as our arm, each step a bounded sample (one image of the batch through the whole
    chain for the YOLO-style workload)."""
    world, rank, local = dist_setup()
    if rank != 0:
        return
    import oracle
    oracle.build()
    from conv_bn_activation_gb300 import synthetic, workloads
    if args.workload == "yolo":
        stages = synthetic.yolo_params()
        x = synthetic.yolo_input(32)
        n = 1

        def step(i):
            h = x[i % 32:i % 32 + n]
            for st in stages:
                h = oracle.yolo_stage(h, st).astype(np.float32)

        unit, per_step, sample = "images/s", n, f"{n} image of the 32-image batch per step, all 20 layers"
        config = {"workload": "YOLO-style 20-conv chain (5 stages, concat via channel views, post-act residual), "
                              "640x640x3 fp32", "batch": 32, "l2": "n/a (CPU)"}
    elif args.workload == "depthwise":
        xd, w, bn = synthetic.depthwise_layer()
        wl = workloads.depthwise_workload()
        n = 1

        def step(i):
            xs = xd[i % 64:i % 64 + n]
            oracle.conv_bn_act(xs, w, bn, stride=1, pad=1, groups=384, act=oracle.ACT_RELU)
            oracle.conv_bn_act(xs, w, bn, stride=2, pad=1, groups=384, act=oracle.ACT_RELU)

        unit, per_step = "GB/s", (wl["s1"].bytes + wl["s2"].bytes) * n / 64 / 1e9
        sample = f"{n} image of the 64-image batch per step, stride 1 and 2"
        config = {"workload": "depthwise 3x3 + BN + ReLU, NHWC fp32, N=64 C=384 56x56, stride 1 and 2",
                  "batch": 64, "l2": "n/a (CPU)"}
    else:
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm is timed on the yolo (default) "
                          "and depthwise workloads only"}))
        return
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="yolo", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of one captured graph")
    ap.add_argument("--launch-reps", type=int, default=20, help="back-to-back repetitions per kernel timing")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="passes per step are scaled so that the K timed steps last at least this long")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="default (yolo) run: skip the other configurations measured beside it")
    ap.add_argument("--profile-pass", action="store_true",
                    help="set up, warm up, run one pass inside the NVTX range 'profiled_pass' and exit (profilers)")
    ap.add_argument("--no-autotune", action="store_true",
                    help="dense / yolo: keep the built-in tile cost model instead of measuring plans at setup")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
