"""GPU parity of the 8 -> 8 channel 3x3 stride-1 kernel (conv3x3_c8.cu) against the fp64 oracle.

The kernel keeps 34 x 34 input pixels per 32 x 32 output tile in shared memory and accumulates the
even and odd input channels in separate halves of packed FMAs; it is fp32 throughout, so the bar
is 1e-5 relative to max|oracle|.  Shapes cover tiles cut by the image edge on every side (images
narrower and shorter than a tile, one pixel, sizes one past a tile), several images, every
epilogue variant, the YOLO-style chain's channel-slice views (input and output inside 16-channel
pixels) with padded output rows whose padding must survive, and views the kernel must leave to
the generic direct kernel.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(1, 1, 1), (1, 32, 32), (2, 33, 33), (1, 5, 70), (3, 70, 5), (2, 31, 97), (1, 64, 31), (1, 320, 320)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_c8_shapes(gpu, orc, shape):
    N, H, W = shape
    x, w, bn = synthetic.dense_layer(8, 8, H, W, N=N, k=3, seed=H * 7 + W)
    layer = ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)
    y = torch.empty(N, H, W, 8, device=gpu)
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_DIRECT
    layer(xd, y)
    sync_check()
    assert "conv3x3_c8" in cb.last_launch()["kernel"]
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 0), (2, 0), (1, 1), (2, 2), (0, 2), (2, 1)])
def test_c8_epilogue_variants(gpu, orc, act, res_mode):
    N, H, W = 2, 37, 45
    x, w, bn = synthetic.dense_layer(8, 8, H, W, N=N, k=3, seed=act * 3 + res_mode)
    r = np.random.default_rng(act + 10 * res_mode).standard_normal((N, H, W, 8)).astype(np.float32)
    y = torch.empty(N, H, W, 8, device=gpu)
    ConvBnAct(w, bn, 1, 1, act)(to_dev(x), y, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_c8_channel_slice_views_and_padded_rows(gpu, orc):
    """As in the chain: x = the first 8 channels of a 16-channel buffer, y = the last 8 channels of
    another, whose rows are padded; channels and columns outside y keep their canaries."""
    N, H, W = 2, 40, 50
    x, w, bn = synthetic.dense_layer(8, 8, H, W, N=N, k=3, seed=3)
    xbuf = torch.zeros(N, H, W, 16, device=gpu)
    xbuf[..., :8] = to_dev(x)
    xbuf[..., 8:] = 1e6                                    # must not leak into the result
    ybuf = canary_buffer((N, H, W + 6, 16))
    y = ybuf[:, :, :W, 8:]
    ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)(xbuf[..., :8], y)
    sync_check()
    assert is_canary(ybuf[:, :, :W, :8]) and is_canary(ybuf[:, :, W:, :])
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_c8_unaligned_views_take_the_generic_kernel(gpu, orc):
    """Pixels 36 bytes apart (9 channels per pixel) cannot be copied in 16-byte pieces: the layer
    still runs, on the generic direct kernel, and still matches."""
    N, H, W = 1, 20, 21
    x, w, bn = synthetic.dense_layer(8, 8, H, W, N=N, k=3, seed=9)
    xbuf = torch.zeros(N, H, W, 9, device=gpu)
    xbuf[..., :8] = to_dev(x)
    y = torch.empty(N, H, W, 8, device=gpu)
    ConvBnAct(w, bn, 1, 1, cb.ACT_RELU)(xbuf[..., :8], y)
    sync_check()
    assert "conv3x3_c8" not in cb.last_launch()["kernel"]
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_RELU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 33, 33), (1, 5, 70), (3, 70, 5), (2, 64, 31)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("act,res_mode", [(2, 0), (1, 1), (2, 2)])
def test_c8_bf16(gpu, orc, shape, act, res_mode):
    """bf16 storage (x, y, residual bf16; fp32 weights and arithmetic): within half a bf16 ulp of the
    oracle on the same bf16 values, and bit-equal to the fp32 kernel's output rounded to bf16 (the
    two run the same fp32 sums)."""
    from gpu_util import bf16_within_half_ulp, to_dev_bf16
    N, H, W = shape
    x, w, bn = synthetic.dense_layer(8, 8, H, W, N=N, k=3, seed=H + W + act)
    r = np.random.default_rng(res_mode).standard_normal((N, H, W, 8)).astype(np.float32)
    xd, xv = to_dev_bf16(x)
    rd, rv = to_dev_bf16(r)
    layer = ConvBnAct(w, bn, 1, 1, act)
    y = torch.empty(N, H, W, 8, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_DIRECT
    layer(xd, y, residual=rd if res_mode else None, res_mode=res_mode)
    sync_check()
    assert "conv3x3_c8" in cb.last_launch()["kernel"]
    ref = orc.conv_bn_act(xv, w, bn, stride=1, pad=1, act=act, residual=rv if res_mode else None, res_mode=res_mode)
    assert bf16_within_half_ulp(y.float().cpu().numpy(), ref) <= 1.0
    y32 = torch.empty(N, H, W, 8, device=gpu)
    layer(torch.from_numpy(xv).to(gpu), y32, residual=torch.from_numpy(rv).to(gpu) if res_mode else None,
          res_mode=res_mode)
    sync_check()
    assert torch.equal(y.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
