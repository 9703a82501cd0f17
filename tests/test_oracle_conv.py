"""Pins for the oracle's convolution (CPU only).

The oracle is a direct 7-loop convolution with zero padding and window origin
(oh*s - p, ow*s - p) ("How I sped up convolutions", Metal kernel steps 2-3).
Each check below ties it to something other than itself: a hand-computed
example, an independent im2col + matmul formulation, PyTorch's CPU conv2d in
float64, and invariants (identity kernel, 1x1 = matmul, stride-2 = strided
stride-1, depthwise = block-diagonal dense, linearity).
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

pytestmark = pytest.mark.filterwarnings("ignore")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _im2col_conv(x_nhwc, w_oihw, s, p, groups):
    """Independent formulation: pad, gather windows, one matmul per group (fp64)."""
    x = np.asarray(x_nhwc, dtype=np.float64)
    w = np.asarray(w_oihw, dtype=np.float64)
    N, H, W, C = x.shape
    Co, cg, kh, kw = w.shape
    OH, OW = (H + 2 * p - kh) // s + 1, (W + 2 * p - kw) // s + 1
    xp = np.zeros((N, H + 2 * p, W + 2 * p, C))
    xp[:, p:p + H, p:p + W, :] = x
    cols = np.empty((N, OH, OW, kh, kw, C))
    for i in range(kh):
        for j in range(kw):
            cols[:, :, :, i, j, :] = xp[:, i:i + s * (OH - 1) + 1:s, j:j + s * (OW - 1) + 1:s, :]
    out = np.empty((N, OH, OW, Co))
    og = Co // groups
    for g in range(groups):
        a = cols[..., g * cg:(g + 1) * cg].transpose(0, 1, 2, 5, 3, 4).reshape(N * OH * OW, cg * kh * kw)
        b = w[g * og:(g + 1) * og].reshape(og, cg * kh * kw)
        out[..., g * og:(g + 1) * og] = (a @ b.T).reshape(N, OH, OW, og)
    return out


def _torch_conv(x_nhwc, w_oihw, s, p, groups):
    x = torch.from_numpy(np.ascontiguousarray(x_nhwc, dtype=np.float64)).permute(0, 3, 1, 2)
    w = torch.from_numpy(np.asarray(w_oihw, dtype=np.float64))
    return F.conv2d(x, w, stride=s, padding=p, groups=groups).permute(0, 2, 3, 1).numpy()


def test_hand_computed_example(orc):
    """3x3 image 1..9, all-ones 3x3 kernel, pad 1: values summed by hand (golden file)."""
    g = json.load(open(os.path.join(GOLDEN, "conv_hand_example.json")))
    x = np.array(g["x"], dtype=np.float32).reshape(1, 3, 3, 1)
    w = np.ones((1, 1, 3, 3), dtype=np.float32)
    z = orc.conv2d(x, w, stride=1, pad=1)[0, :, :, 0]
    np.testing.assert_array_equal(z, np.array(g["stride1_pad1"], dtype=np.float64))
    z2 = orc.conv2d(x, w, stride=2, pad=1)[0, :, :, 0]
    np.testing.assert_array_equal(z2, np.array(g["stride2_pad1"], dtype=np.float64))
    z0 = orc.conv2d(x, w, stride=1, pad=0)[0, :, :, 0]
    np.testing.assert_array_equal(z0, np.array(g["stride1_pad0"], dtype=np.float64))


CASES = [
    # N, H, W, C, Co, k, s, p, groups
    (2, 7, 5, 3, 4, 3, 1, 1, 1),
    (1, 8, 9, 4, 6, 3, 2, 1, 1),
    (2, 6, 6, 5, 5, 3, 1, 1, 5),
    (1, 9, 7, 8, 8, 3, 2, 1, 8),
    (3, 5, 4, 6, 7, 1, 1, 0, 1),
    (1, 6, 7, 4, 3, 1, 2, 0, 1),
    (1, 4, 4, 1, 3, 3, 1, 0, 1),
    (2, 5, 6, 6, 4, 3, 1, 1, 2),
]


@pytest.mark.parametrize("case", CASES)
def test_conv_vs_im2col_and_torch(orc, case):
    N, H, W, C, Co, k, s, p, groups = case
    g = np.random.default_rng(hash(case) % 2**32)
    x = g.standard_normal((N, H, W, C)).astype(np.float32)
    w = g.standard_normal((Co, C // groups, k, k)).astype(np.float32)
    z = orc.conv2d(x, w, stride=s, pad=p, groups=groups)
    np.testing.assert_allclose(z, _im2col_conv(x, w, s, p, groups), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(z, _torch_conv(x, w, s, p, groups), rtol=1e-12, atol=1e-12)


def test_nchw_input_matches_nhwc(orc):
    g = np.random.default_rng(5)
    x = g.standard_normal((2, 7, 9, 3)).astype(np.float32)
    w = g.standard_normal((4, 3, 3, 3)).astype(np.float32)
    a = orc.conv2d(x, w, stride=2, pad=1)
    b = orc.conv2d(np.ascontiguousarray(x.transpose(0, 3, 1, 2)), w, stride=2, pad=1, layout=orc.NCHW)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("groups", [1, 6])
def test_identity_kernel(orc, groups):
    """Centre tap 1, pad 1, stride 1 (diagonal for dense) reproduces the input exactly."""
    g = np.random.default_rng(6)
    C = 6
    x = g.standard_normal((2, 5, 7, C)).astype(np.float32)
    if groups == 1:
        w = np.zeros((C, C, 3, 3), np.float32)
        for c in range(C):
            w[c, c, 1, 1] = 1
    else:
        w = np.zeros((C, 1, 3, 3), np.float32)
        w[:, 0, 1, 1] = 1
    np.testing.assert_array_equal(orc.conv2d(x, w, stride=1, pad=1, groups=groups), x.astype(np.float64))


def test_pointwise_is_matmul(orc):
    g = np.random.default_rng(7)
    x = g.standard_normal((2, 4, 5, 8)).astype(np.float32)
    w = g.standard_normal((3, 8, 1, 1)).astype(np.float32)
    ref = x.astype(np.float64).reshape(-1, 8) @ w[:, :, 0, 0].astype(np.float64).T
    np.testing.assert_allclose(orc.conv2d(x, w).reshape(-1, 3), ref, rtol=1e-13, atol=1e-13)


def test_stride2_is_subsampled_stride1(orc):
    g = np.random.default_rng(8)
    x = g.standard_normal((1, 9, 8, 4)).astype(np.float32)
    w = g.standard_normal((5, 4, 3, 3)).astype(np.float32)
    z1 = orc.conv2d(x, w, stride=1, pad=1)
    z2 = orc.conv2d(x, w, stride=2, pad=1)
    np.testing.assert_array_equal(z2, z1[:, ::2, ::2, :])


def test_depthwise_is_block_diagonal_dense(orc):
    g = np.random.default_rng(9)
    C = 5
    x = g.standard_normal((2, 6, 7, C)).astype(np.float32)
    wd = g.standard_normal((C, 1, 3, 3)).astype(np.float32)
    wf = np.zeros((C, C, 3, 3), np.float32)
    for c in range(C):
        wf[c, c] = wd[c, 0]
    for s in (1, 2):
        np.testing.assert_allclose(orc.conv2d(x, wd, stride=s, pad=1, groups=C),
                                   orc.conv2d(x, wf, stride=s, pad=1), rtol=1e-14, atol=1e-14)


def test_linearity(orc):
    g = np.random.default_rng(10)
    x1 = g.standard_normal((1, 5, 6, 3)).astype(np.float32)
    x2 = g.standard_normal((1, 5, 6, 3)).astype(np.float32)
    w1 = g.standard_normal((4, 3, 3, 3)).astype(np.float32)
    w2 = g.standard_normal((4, 3, 3, 3)).astype(np.float32)
    # conv(x1 + x2, w) with the sum formed exactly in fp64 through two calls
    np.testing.assert_allclose(orc.conv2d(x1, w1, pad=1) + orc.conv2d(x2, w1, pad=1),
                               _im2col_conv(x1.astype(np.float64) + x2, w1, 1, 1, 1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.conv2d(x1, w1, pad=1) + orc.conv2d(x1, w2, pad=1),
                               _im2col_conv(x1, w1.astype(np.float64) + w2, 1, 1, 1), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.conv2d(2 * x1, w1, pad=1), 2 * orc.conv2d(x1, w1, pad=1), rtol=0, atol=0)


def test_padding_only_touches_border(orc):
    """With pad 1 the interior equals the unpadded (valid) convolution."""
    g = np.random.default_rng(11)
    x = g.standard_normal((1, 7, 8, 3)).astype(np.float32)
    w = g.standard_normal((2, 3, 3, 3)).astype(np.float32)
    np.testing.assert_array_equal(orc.conv2d(x, w, pad=1)[:, 1:-1, 1:-1], orc.conv2d(x, w, pad=0))


def test_points_match_full(orc):
    g = np.random.default_rng(12)
    x = g.standard_normal((2, 9, 7, 6)).astype(np.float32)
    w = g.standard_normal((6, 1, 3, 3)).astype(np.float32)
    bn = tuple(g.uniform(0.5, 1.5, 6).astype(np.float32) for _ in range(4))
    r = g.standard_normal((2, 5, 4, 6)).astype(np.float32)
    full = orc.conv_bn_act(x, w, bn, stride=2, pad=1, groups=6, act=orc.ACT_SILU, residual=r,
                           res_mode=orc.RES_POST_ACT)
    idx = g.choice(full.size, 50, replace=False)
    pts = orc.conv_bn_act_points(x, w, bn, idx, stride=2, pad=1, groups=6, act=orc.ACT_SILU,
                                 residual=r, res_mode=orc.RES_POST_ACT)
    np.testing.assert_array_equal(pts, full.reshape(-1)[idx])
