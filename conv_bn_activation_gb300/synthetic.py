"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no convolution, normalisation, resize or layout change),
so feeding its arrays to both the CUDA path and the CPU oracle couples them
only through their inputs.

Distributions (one numpy PCG64 generator per workload, seed 1000 + index):
  * BatchNorm: gamma, var ~ U[0.5, 1.5]; beta, mean ~ N(0, 0.1) (std 0.1);
    eps = 1e-5.
  * Kaiming-normal weights: std = sqrt(2 / fan_in), fan_in = (Cin/groups)*kh*kw.
  * "N(0, 1/9)" depthwise weights: variance 1/9, i.e. std 1/3.
Weights are drawn in PyTorch's OIHW layout [Co, Cin/groups, kh, kw];
activations are drawn channel-last (NHWC) except where a workload says NCHW.
"""
from __future__ import annotations

import numpy as np

BN_EPS = 1e-5
SEED_BASE = 1000

# DepthwiseMNIST stages: (Cin, Cout, stride)
MNIST_BLOCKS = ((48, 96, 2), (96, 96, 1), (96, 192, 2), (192, 192, 1))

# Dense 3x3 sweep: (Cin, Cout, H_in, stride)
DENSE_SWEEP = (
    (3, 16, 640, 2), (16, 32, 320, 2), (32, 64, 160, 2), (64, 128, 80, 2), (128, 256, 40, 2),
    (64, 64, 80, 1), (128, 128, 40, 1), (256, 256, 20, 1),
)

# YOLO-style chain: per stage the entry conv's (Cin, Cout)
YOLO_STAGES = ((3, 16), (16, 32), (32, 64), (64, 128), (128, 256))


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def bn_params(g: np.random.Generator, C: int):
    gamma = g.uniform(0.5, 1.5, C).astype(np.float32)
    beta = (g.standard_normal(C) * 0.1).astype(np.float32)
    mean = (g.standard_normal(C) * 0.1).astype(np.float32)
    var = g.uniform(0.5, 1.5, C).astype(np.float32)
    return gamma, beta, mean, var


def kaiming(g: np.random.Generator, co: int, cin_g: int, kh: int, kw: int) -> np.ndarray:
    std = np.sqrt(2.0 / (cin_g * kh * kw))
    return (g.standard_normal((co, cin_g, kh, kw)) * std).astype(np.float32)


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def uniform01(g: np.random.Generator, shape) -> np.ndarray:
    return g.random(shape, dtype=np.float32)


def frames_u8(g: np.random.Generator, shape) -> np.ndarray:
    return g.integers(0, 256, size=shape, dtype=np.uint8)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
def mnist_params(seed: int = SEED_BASE + 0):
    """DepthwiseMNIST: stem 1->48, four depthwise-separable blocks, fc 192->10."""
    g = rng(seed)
    p = {"stem_w": kaiming(g, 48, 1, 3, 3), "stem_bn": bn_params(g, 48), "blocks": []}
    for cin, cout, s in MNIST_BLOCKS:
        blk = {
            "dw_w": kaiming(g, cin, 1, 3, 3), "bn1": bn_params(g, cin),
            "pw_w": kaiming(g, cout, cin, 1, 1), "bn2": bn_params(g, cout),
        }
        if s != 1 or cin != cout:
            blk["skip_w"] = kaiming(g, cout, cin, 1, 1)
            blk["skip_bn"] = bn_params(g, cout)
        p["blocks"].append(blk)
    p["fc_w"] = (g.standard_normal((10, 192)) * np.sqrt(2.0 / 192)).astype(np.float32)
    p["fc_b"] = np.zeros(10, dtype=np.float32)
    return p


def mnist_input(batch: int = 64, seed: int = SEED_BASE + 0):
    """NHWC [batch, 28, 28, 1] ~ U[0, 1] (drawn from a stream separate from the weights)."""
    return uniform01(rng(seed + 100), (batch, 28, 28, 1))


def depthwise_layer(N=64, C=384, H=56, W=56, seed: int = SEED_BASE + 1):
    """Depthwise 3x3 layer: x ~ N(0,1) NHWC, w ~ N(0, 1/9), BN as the MNIST net."""
    g = rng(seed)
    w = normal(g, (C, 1, 3, 3), std=1.0 / 3.0)
    bn = bn_params(g, C)
    x = normal(g, (N, H, W, C))
    return x, w, bn


def dense_layer(cin, cout, H, W=None, N=1, k=3, seed: int = SEED_BASE + 2):
    """Dense conv layer: x ~ N(0,1) NHWC, Kaiming weights, BN."""
    W = H if W is None else W
    g = rng(seed + 7919 * cin + 104729 * cout + H)
    w = kaiming(g, cout, cin, k, k)
    bn = bn_params(g, cout)
    x = normal(g, (N, H, W, cin))
    return x, w, bn


def yolo_params(seed: int = SEED_BASE + 3):
    """Five stages: entry 3x3 s2 (Cin->C), 1x1 C->C/2, 3x3 C/2->C/2, 1x1 C->C."""
    g = rng(seed)
    stages = []
    for cin, c in YOLO_STAGES:
        h = c // 2
        stages.append({
            "down_w": kaiming(g, c, cin, 3, 3), "down_bn": bn_params(g, c),
            "cv1_w": kaiming(g, h, c, 1, 1), "cv1_bn": bn_params(g, h),
            "cv2_w": kaiming(g, h, h, 3, 3), "cv2_bn": bn_params(g, h),
            "cv3_w": kaiming(g, c, c, 1, 1), "cv3_bn": bn_params(g, c),
        })
    return stages


def yolo_input(batch: int, size: int = 640, seed: int = SEED_BASE + 3):
    return uniform01(rng(seed + 100), (batch, size, size, 3))


def preprocess_frames(N=32, H=720, W=1280, seed: int = SEED_BASE + 4):
    """u8 HWC frames ~ U{0..255}."""
    return frames_u8(rng(seed), (N, H, W, 3))


def stem_params(seed: int = SEED_BASE + 4):
    """Stem conv 3->16, 3x3, stride 2, + BN (fed by the preprocess)."""
    g = rng(seed + 100)
    return kaiming(g, 16, 3, 3, 3), bn_params(g, 16)
