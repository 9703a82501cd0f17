"""Pins for the oracle's u8 frame preprocess (CPU only).

Definition ("A fused Ampere preprocess kernel": the byte ledger and "bilinear
is a contract"; OpenCV half-pixel convention): f = (d + 0.5) * S/D - 0.5,
i0 = floor(f), a = f - i0, clamped at both borders; bilinear value rounded
half up to u8; u8 / 255 in fp32; planar (NCHW) output.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from conv_bn_activation_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _exact_coords(S, D):
    """Exact rational sample coordinates (Python fractions), with the border rules."""
    i0s, i1s, As = [], [], []
    for d in range(D):
        f = (Fraction(2 * d + 1, 2)) * Fraction(S, D) - Fraction(1, 2)
        k = f.numerator // f.denominator
        a = f - k
        if k < 0:
            k, a = 0, Fraction(0)
        if k >= S - 1:
            k, a = S - 1, Fraction(0)
        i0s.append(k)
        i1s.append(min(k + 1, S - 1))
        As.append(a)
    return i0s, i1s, As


SIZES = [(1280, 640), (720, 480), (13, 7), (7, 13), (100, 37), (37, 100), (5, 5), (64, 16), (3, 8), (1, 4)]


@pytest.mark.parametrize("S,D", SIZES)
def test_coords_match_exact_rationals(orc, S, D):
    i0, i1, a = orc.axis_coords(S, D, orc.PREC_F64)
    e0, e1, ea = _exact_coords(S, D)
    np.testing.assert_array_equal(i0, e0)
    np.testing.assert_array_equal(i1, e1)
    np.testing.assert_allclose(a, [float(t) for t in ea], rtol=0, atol=1e-12)


def test_workload_ratio_weights(orc):
    """1280x720 -> 640x480: x weights are exactly 1/2, y weights alternate 1/4, 3/4."""
    i0, i1, ax = orc.axis_coords(1280, 640, orc.PREC_F64)
    assert np.all(ax == 0.5) and np.array_equal(i0, 2 * np.arange(640)) and np.array_equal(i1, i0 + 1)
    j0, j1, ay = orc.axis_coords(720, 480, orc.PREC_F64)
    np.testing.assert_array_equal(ay, np.where(np.arange(480) % 2 == 0, 0.25, 0.75))
    np.testing.assert_array_equal(j0, (3 * np.arange(480) + 1) // 2 - (np.arange(480) % 2 == 1))
    # fp32 coordinates are exact at this ratio
    for S, D in ((1280, 640), (720, 480)):
        a64 = orc.axis_coords(S, D, orc.PREC_F64)
        a32 = orc.axis_coords(S, D, orc.PREC_F32)
        for u, v in zip(a64, a32):
            np.testing.assert_array_equal(u, v)


def test_constant_frame(orc):
    for v in (0, 1, 127, 128, 254, 255):
        src = np.full((2, 9, 11, 3), v, np.uint8)
        out = orc.preprocess_u8(src, 5, 7)
        assert out.shape == (2, 3, 5, 7)
        assert np.all(out == np.float32(v) / np.float32(255))


def test_ramp_frame_is_reproduced_at_sample_points(orc):
    """Bilinear interpolation of p = x + 2y is exact: v = fx + 2 fy where unclamped."""
    Hs, Ws, Hd, Wd = 40, 60, 17, 23
    yy, xx = np.meshgrid(np.arange(Hs), np.arange(Ws), indexing="ij")
    ramp = (xx + 2 * yy)
    assert ramp.max() <= 255
    src = np.repeat(ramp[None, :, :, None], 3, axis=3).astype(np.uint8)
    _, v = orc.resize_u8(src, Hd, Wd, return_values=True)
    fx = (np.arange(Wd) + 0.5) * Ws / Wd - 0.5
    fy = (np.arange(Hd) + 0.5) * Hs / Hd - 0.5
    okx = (fx >= 0) & (fx <= Ws - 1)
    oky = (fy >= 0) & (fy <= Hs - 1)
    want = fx[None, :] + 2 * fy[:, None]
    got = v[0, :, :, 0]
    m = oky[:, None] & okx[None, :]
    np.testing.assert_allclose(got[m], want[m], rtol=0, atol=1e-9)


def test_same_size_is_identity(orc):
    src = np.random.default_rng(1).integers(0, 256, (2, 6, 9, 3), dtype=np.uint8)
    np.testing.assert_array_equal(orc.resize_u8(src, 6, 9), src)
    out = orc.preprocess_u8(src, 6, 9)
    np.testing.assert_array_equal(out, src.transpose(0, 3, 1, 2).astype(np.float32) / np.float32(255))


def test_values_match_torch_bilinear(orc):
    """PyTorch's bilinear (align_corners=False) uses the same half-pixel rule: compare unrounded values."""
    g = np.random.default_rng(2)
    for (Hs, Ws, Hd, Wd) in ((720, 1280, 480, 640), (31, 45, 17, 20), (10, 12, 25, 31)):
        src = g.integers(0, 256, (1, Hs, Ws, 3), dtype=np.uint8)
        _, v = orc.resize_u8(src, Hd, Wd, return_values=True)
        t = torch.from_numpy(src.astype(np.float64)).permute(0, 3, 1, 2)
        ref = F.interpolate(t, size=(Hd, Wd), mode="bilinear", align_corners=False).permute(0, 2, 3, 1).numpy()
        np.testing.assert_allclose(v, ref, rtol=0, atol=1e-9)


def test_round_half_up(orc):
    """Two pixels 0 and 1 with weight 1/2 each give v = 0.5, which rounds up to 1."""
    src = np.zeros((1, 1, 4, 3), np.uint8)
    src[0, 0, 1, :] = 1          # row: 0 1 0 0
    out, v = orc.resize_u8(src, 1, 2, return_values=True)   # fx = 2dx + 0.5
    assert v[0, 0, 0, 0] == 0.5 and out[0, 0, 0, 0] == 1
    src[0, 0, 1, :] = 2          # 1.0 exactly
    out, v = orc.resize_u8(src, 1, 2, return_values=True)
    assert v[0, 0, 0, 0] == 1.0 and out[0, 0, 0, 0] == 1


def test_three_pass_equals_fused(orc):
    src = np.random.default_rng(3).integers(0, 256, (2, 72, 128, 3), dtype=np.uint8)
    for prec in (orc.PREC_F64, orc.PREC_F32):
        np.testing.assert_array_equal(orc.preprocess_u8_three_pass(src, 48, 64, prec),
                                      orc.preprocess_u8(src, 48, 64, prec))


def test_f32_decision_equals_f64_at_dyadic_ratios(orc):
    g = np.random.default_rng(4)
    for (Hs, Ws, Hd, Wd) in ((72, 128, 48, 64), (36, 40, 48, 32), (16, 16, 4, 8)):
        src = g.integers(0, 256, (2, Hs, Ws, 3), dtype=np.uint8)
        np.testing.assert_array_equal(orc.preprocess_u8(src, Hd, Wd, orc.PREC_F32),
                                      orc.preprocess_u8(src, Hd, Wd, orc.PREC_F64))


def test_f32_decision_differs_only_at_near_ties(orc):
    """At a non-dyadic ratio the fp32 and fp64 u8 codes differ by at most 1, only where v is near x.5."""
    src = np.random.default_rng(5).integers(0, 256, (1, 100, 100, 3), dtype=np.uint8)
    u64, v64 = orc.resize_u8(src, 37, 41, orc.PREC_F64, return_values=True)
    u32 = orc.resize_u8(src, 37, 41, orc.PREC_F32)
    d = u64.astype(int) - u32.astype(int)
    assert np.abs(d).max() <= 1
    frac = v64 - np.floor(v64)
    assert np.all(np.abs(frac[d != 0] - 0.5) < 1e-3)


def test_byte_ledger_matches_page():
    """The per-pass ledger and the fused/unfused ratio printed on the page (MB = 1e6 B)."""
    g = json.load(open(os.path.join(GOLDEN, "preprocess_ledger.json")))
    fr = g["frame"]
    led = workloads.preprocess_ledger(fr["src_h"], fr["src_w"], fr["dst_h"], fr["dst_w"])
    mb = g["ledger_mb"]
    p = led["passes"]
    assert round(p["resize"] / 1e6, 2) == mb["resize_total"]
    assert round(p["normalize"] / 1e6, 2) == mb["normalize_total"]
    assert round(p["layout"] / 1e6, 2) == mb["layout_total"]
    assert round(led["unfused"] / 1e6, 2) == mb["unfused_total"]
    assert round(led["fused"] / 1e6, 2) == mb["fused_total"]
    assert led["unfused"] == 15_667_200 and led["fused"] == 6_451_200
    assert round(led["unfused"] / led["fused"], 2) == g["predicted_ratio"]
    m = g["measured"]
    # the page's GB/s is ledger bytes / mean time
    assert abs(led["unfused"] / (m["path_a_mean_us"] * 1e-6) / 1e9 - m["path_a_gbps"]) < 0.01
    assert abs(led["fused"] / (m["path_b_mean_us"] * 1e-6) / 1e9 - m["path_b_gbps"]) < 0.01
    assert round(m["path_a_mean_us"] / m["path_b_mean_us"], 3) == m["speedup"]


def test_preprocess_stem_ledger():
    """The fused preprocess + stem moves the u8 frame in and the stem's 16-channel fp32 output out:
    the fused preprocess's ledger minus its fp32 planar write, plus the stem output (half the
    resolution in each direction, 16 channels), weights and scale/bias once."""
    led = workloads.preprocess_ledger(720, 1280, 480, 640)
    planar = 480 * 640 * 3 * 4
    stem_out = 240 * 320 * 16 * 4
    w = workloads.preprocess_stem_fused(32, 720, 1280, 480, 640)
    assert w.bytes == 32 * (led["fused"] - planar + stem_out) + (16 * 27 + 2 * 16) * 4
    assert w.flops == 2 * 32 * 240 * 320 * 16 * 27
