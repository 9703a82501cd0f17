"""GPU parity of the streaming CUDA-core 1x1 kernel (stride 1, Ci and Co in {4, 8, 16, 32}).

It computes in fp32 (no TF32 rounding), so the bar is the CUDA-core one: 1e-5 of max|oracle|.
Covered: every (Ci, Co) pair it takes, the epilogue variants, channel-slice input and output views
(the YOLO concat), padded rows (canaries must survive, and the non-flat addressing runs), the
in-place residual, and the shapes it must not take.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

CH = [4, 8, 16, 32]


@pytest.mark.parametrize("ci", CH)
@pytest.mark.parametrize("co", CH)
def test_pointwise_channels(gpu, orc, ci, co):
    x, w, bn = synthetic.dense_layer(ci, co, 13, 17, N=3, k=1, seed=ci * 100 + co)
    layer = ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)
    assert not layer.tc_weights
    xd = to_dev(x)
    y = torch.empty(3, 13, 17, co, device="cuda")
    assert cb.conv_path(xd, y, 1, 1, 0) == cb.PATH_POINTWISE
    layer(xd, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), orc.conv_bn_act(x, w, bn, stride=1, pad=0, act=orc.ACT_SILU)) <= TOL_FP32


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 0), (1, 1), (2, 2), (0, 2), (2, 1)])
def test_pointwise_epilogues(gpu, orc, act, res_mode):
    x, w, bn = synthetic.dense_layer(16, 16, 20, 9, N=2, k=1, seed=act + 3 * res_mode)
    r = np.random.default_rng(8).standard_normal((2, 20, 9, 16)).astype(np.float32)
    layer = ConvBnAct(w, bn, 1, 0, act)
    y = torch.empty(2, 20, 9, 16, device="cuda")
    layer(to_dev(x), y, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=0, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_pointwise_channel_slices_and_padded_rows(gpu, orc):
    """x is a channel slice of a wider buffer, y a slice of a padded one (non-flat pixel
    addressing); every element outside y's view keeps its canary."""
    N, H, W, ci, co = 2, 11, 14, 8, 16
    x, w, bn = synthetic.dense_layer(ci, co, H, W, N=N, k=1, seed=21)
    xbuf = torch.randn(N, H, W, ci + 8, device="cuda")
    xbuf[..., 4:4 + ci] = to_dev(x)
    xv = xbuf[..., 4:4 + ci]
    ybuf = canary_buffer((N, H, W + 2, co + 8))
    yv = ybuf[:, :, :W, 8:8 + co]
    layer = ConvBnAct(w, bn, 1, 0, cb.ACT_RELU)
    assert cb.conv_path(xv, yv, 1, 1, 0) == cb.PATH_POINTWISE
    layer(xv, yv)
    sync_check()
    assert rel_err(yv.cpu().numpy(), orc.conv_bn_act(x, w, bn, stride=1, pad=0, act=orc.ACT_RELU)) <= TOL_FP32
    assert is_canary(ybuf[:, :, W:, :]) and is_canary(ybuf[:, :, :W, :8])


def test_pointwise_inplace_residual(gpu, orc):
    x, w, bn = synthetic.dense_layer(32, 32, 10, 10, N=2, k=1, seed=22)
    r = np.random.default_rng(9).standard_normal((2, 10, 10, 32)).astype(np.float32)
    y = to_dev(r)
    ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)(to_dev(x), y, residual=y, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=0, act=orc.ACT_SILU, residual=r, res_mode=orc.RES_POST_ACT)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_pointwise_not_taken_outside_its_shapes(gpu):
    x = torch.empty(1, 4, 4, 48, device="cuda")
    assert cb.conv_path(x, torch.empty(1, 4, 4, 16, device="cuda"), 1, 1, 0) == cb.PATH_TC_IM2COL
    x = torch.empty(1, 4, 4, 16, device="cuda")
    assert cb.conv_path(x, torch.empty(1, 4, 4, 24, device="cuda"), 1, 1, 0) == cb.PATH_TC_IM2COL
    assert cb.conv_path(x, torch.empty(1, 2, 2, 16, device="cuda"), 1, 2, 0) == cb.PATH_TC_IM2COL
    cb.set_kernel_policy(1)
    try:
        assert cb.conv_path(x, torch.empty(1, 4, 4, 16, device="cuda"), 1, 1, 0) == cb.PATH_DIRECT
    finally:
        cb.set_kernel_policy(0)


@pytest.mark.parametrize("ci,co", [(4, 32), (8, 32), (32, 4)])
def test_pointwise_residual_extreme_widths(gpu, orc, ci, co):
    """Residual tiles for the widest output per input channel (the 4 -> 32 ring does not fit in
    shared memory and runs on the direct kernel instead)."""
    x, w, bn = synthetic.dense_layer(ci, co, 9, 31, N=2, k=1, seed=ci + co)
    r = np.random.default_rng(10).standard_normal((2, 9, 31, co)).astype(np.float32)
    y = torch.empty(2, 9, 31, co, device="cuda")
    ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)(to_dev(x), y, residual=to_dev(r), res_mode=cb.RES_PRE_ACT)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=0, act=orc.ACT_SILU, residual=r, res_mode=orc.RES_PRE_ACT)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32
