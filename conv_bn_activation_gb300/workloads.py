"""Algorithmic bytes and FLOPs of each step of the hot path (the roofline numerators).

"Algorithmic" means compulsory DRAM traffic: every input element read once,
every output element written once, weights and per-channel scale/bias read
once.  Halo re-reads, partial-sector traffic and L2 misses are not counted;
measured DRAM traffic above these figures is waste.

The preprocess ledger follows "A fused Ampere preprocess kernel" (the byte
ledger per pass): the resize reads the u8 frame and writes a u8 resized frame,
the normalize reads it and writes fp32, the layout pass reads and writes fp32;
the fused pass reads the u8 frame once and writes the fp32 planar tensor once.
FLOPs count one multiply and one add per multiply-accumulate of the
convolution only (BN, activation and residual are not counted), which is the
convention behind the depthwise arithmetic intensities quoted on "How I sped
up convolutions" (about 0.87-2.2 FLOP/byte for its depthwise layers).
"""
from __future__ import annotations

from dataclasses import dataclass

F32 = 4


def out_size(n: int, k: int, s: int, p: int) -> int:
    return (n + 2 * p - k) // s + 1


@dataclass(frozen=True)
class Work:
    bytes: int
    flops: int

    @property
    def intensity(self) -> float:
        return self.flops / self.bytes if self.bytes else 0.0

    def __add__(self, other: "Work") -> "Work":
        return Work(self.bytes + other.bytes, self.flops + other.flops)


def conv_layer(N, H, W, Cin, Cout, k, s, p, groups=1, residual=False, act_bytes=F32, w_bytes=F32) -> Work:
    """Fused conv + folded BN (+ residual) + activation: in + out (+ r) + w + scale/bias.
    act_bytes: bytes per activation element (4 fp32, 2 bf16 storage); w_bytes: bytes per weight
    (4, or 2 for bf16 tensor-core layers, which multiply bf16 weights)."""
    OH, OW = out_size(H, k, s, p), out_size(W, k, s, p)
    x = N * H * W * Cin * act_bytes
    y = N * OH * OW * Cout * act_bytes
    w = Cout * (Cin // groups) * k * k * w_bytes
    sb = 2 * Cout * F32
    r = y if residual else 0
    macs = N * OH * OW * Cout * (Cin // groups) * k * k
    return Work(x + y + w + sb + r, 2 * macs)


def depthwise_layer(N, H, W, C, s, k=3, p=1, act_bytes=F32) -> Work:
    return conv_layer(N, H, W, C, C, k, s, p, groups=C, act_bytes=act_bytes)


# --- preprocess ledger ("A fused Ampere preprocess kernel", the theory) -----
def preprocess_ledger(Hs, Ws, Hd, Wd, channels=3):
    """Bytes through DRAM per frame for each pass of the unfused path and the fused path."""
    src = Hs * Ws * channels                 # u8 frame
    mid_u8 = Hd * Wd * channels              # u8 resized frame
    f32 = Hd * Wd * channels * F32           # fp32 tensor (HWC or CHW)
    passes = {
        "resize": src + mid_u8,
        "normalize": mid_u8 + f32,
        "layout": f32 + f32,
    }
    return {"passes": passes, "unfused": sum(passes.values()), "fused": src + f32}


def preprocess_fused(N, Hs, Ws, Hd, Wd) -> Work:
    return Work(N * preprocess_ledger(Hs, Ws, Hd, Wd)["fused"], 0)


def preprocess_stem_fused(N, Hs, Ws, Hd, Wd, Cout=16) -> Work:
    """The preprocess fused into the 3x3 stride-2 stem: the u8 frames read once, the stem's fp32
    output written once (plus its weights and scale/bias); FLOPs of the stem convolution."""
    stem = conv_layer(N, Hd, Wd, 3, Cout, 3, 2, 1)
    planar_in = N * Hd * Wd * 3 * F32
    return Work(N * Hs * Ws * 3 + stem.bytes - planar_in, stem.flops)


def preprocess_unfused(N, Hs, Ws, Hd, Wd) -> Work:
    return Work(N * preprocess_ledger(Hs, Ws, Hd, Wd)["unfused"], 0)


# --- whole workloads -------------------------------------------------------
def depthwise_workload(N=64, H=56, W=56, C=384, act_bytes=F32):
    """The depthwise 3x3 + BN + ReLU layer at stride 1 and stride 2."""
    return {"s1": depthwise_layer(N, H, W, C, 1, act_bytes=act_bytes),
            "s2": depthwise_layer(N, H, W, C, 2, act_bytes=act_bytes)}


def mnist_layers(N=64):
    """Per-layer work of the DepthwiseMNIST forward (stem, 4 blocks, pool + fc)."""
    from .synthetic import MNIST_BLOCKS
    layers = [("stem", conv_layer(N, 28, 28, 1, 48, 3, 1, 1))]
    H = 28
    for i, (cin, cout, s) in enumerate(MNIST_BLOCKS):
        OH = out_size(H, 3, s, 1)
        layers.append((f"b{i}.dw", depthwise_layer(N, H, H, cin, s)))
        skip = s != 1 or cin != cout
        layers.append((f"b{i}.pw", conv_layer(N, OH, OH, cin, cout, 1, 1, 0, residual=True)))
        if skip:
            layers.append((f"b{i}.skip", conv_layer(N, H, H, cin, cout, 1, s, 0)))
        H = OH
    pool = Work(N * H * H * 192 * F32 + 10 * 192 * F32 + 10 * F32 + N * 10 * F32,
                N * (H * H * 192 + 2 * 192 * 10))
    layers.append(("pool_fc", pool))
    return layers


def yolo_layers(N=1, size=640, act_bytes=F32, tc_w_bytes=None):
    """Per-layer work of the 20-conv YOLO-style chain.  act_bytes: bytes per activation element;
    tc_w_bytes(cin, cout, k, stride) -> bytes per weight of that layer (default 4)."""
    from .synthetic import YOLO_STAGES
    wb = tc_w_bytes or (lambda ci, co, k, s: F32)
    layers = []
    H = size
    for i, (cin, c) in enumerate(YOLO_STAGES):
        h = c // 2
        OH = out_size(H, 3, 2, 1)
        kw = dict(act_bytes=act_bytes)
        layers.append((f"s{i}.down", conv_layer(N, H, H, cin, c, 3, 2, 1, w_bytes=wb(cin, c, 3, 2), **kw)))
        layers.append((f"s{i}.cv1", conv_layer(N, OH, OH, c, h, 1, 1, 0, w_bytes=wb(c, h, 1, 1), **kw)))
        layers.append((f"s{i}.cv2", conv_layer(N, OH, OH, h, h, 3, 1, 1, w_bytes=wb(h, h, 3, 1), **kw)))
        layers.append((f"s{i}.cv3", conv_layer(N, OH, OH, c, c, 1, 1, 0, residual=True, w_bytes=wb(c, c, 1, 1),
                                               **kw)))
        H = OH
    return layers


def stage_body(N, H, W, C=16, act_bytes=F32) -> Work:
    """The YOLO-style stage body in one kernel (x1 -> out: 1x1 C -> C/2, 3x3 C/2 -> C/2, 1x1 on the
    concat + x1): x1 read once, out written once, the three layers' weights and scale/bias; FLOPs of
    the three convolutions (the 1x1 over the 3x3's halo, recomputed per tile, is not counted)."""
    h = C // 2
    px = N * H * W
    w = (h * C + h * h * 9 + C * C) * F32
    sb = 2 * (h + h + C) * F32
    return Work(2 * px * C * act_bytes + w + sb, 2 * px * (h * C + h * h * 9 + C * C))


def total(layers) -> Work:
    t = Work(0, 0)
    for _, w in layers:
        t = t + w
    return t
