"""GPU parity of the bf16 storage variant: depthwise 3x3 and narrow pointwise 1x1 + folded BN +
activation (+ residual) with x, y and the residual held as bfloat16 and the arithmetic in fp32.

The inputs are bf16 values; the oracle computes in fp64 on exactly those values.  Bars: every
output within half a bf16 unit in the last place of the oracle (2^-8 of the value, plus the
fp32 arithmetic bar), hence within 5e-3 of max|oracle|; and bit-identical to the fp32 kernel's
result on the same inputs rounded to bf16 by torch (the two kernels run the same fp32 sums).
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import (TOL_BF16, bf16_within_half_ulp, canary_buffer_bf16, is_canary_bf16, rel_err, sync_check,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu

SHAPES = [
    # N, H, W, C, stride (C % 8 == 0)
    (2, 9, 13, 32, 1), (2, 9, 13, 32, 2), (3, 14, 14, 48, 2), (2, 7, 7, 192, 1), (1, 5, 130, 64, 1),
    (1, 6, 131, 64, 2), (2, 3, 3, 8, 1), (1, 2, 2, 8, 2), (4, 28, 28, 48, 2), (2, 14, 14, 96, 1),
    (1, 33, 17, 40, 1), (1, 1, 1, 8, 1),
]


def _layer(shape, act, seed):
    N, H, W, C, s = shape
    x, w, bn = synthetic.depthwise_layer(N, C, H, W, seed=seed)
    return x, w, bn, ConvBnAct(w, bn, s, 1, act, groups=C)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bf16_depthwise_relu(gpu, orc, shape):
    N, H, W, C, s = shape
    x, w, bn, layer = _layer(shape, cb.ACT_RELU, seed=sum(shape))
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(H, W)
    y = torch.empty(N, OH, OW, C, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(xd, y, 3, s, 1, groups=C) == cb.PATH_DEPTHWISE
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(xv, w, bn, stride=s, pad=1, groups=C, act=orc.ACT_RELU)
    got = y.float().cpu().numpy()
    assert bf16_within_half_ulp(got, ref) <= 1.0
    assert rel_err(got, ref) <= TOL_BF16


@pytest.mark.parametrize("act,res_mode", [(0, 0), (2, 0), (1, 1), (2, 2), (0, 1), (1, 2)])
@pytest.mark.parametrize("s", [1, 2])
def test_bf16_epilogue_variants(gpu, orc, act, res_mode, s):
    N, H, W, C = 2, 11, 9, 64
    x, w, bn, layer = _layer((N, H, W, C, s), act, seed=7 + act + 3 * res_mode + s)
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(H, W)
    r = np.random.default_rng(3).standard_normal((N, OH, OW, C)).astype(np.float32)
    rd, rv = to_dev_bf16(r)
    y = torch.empty(N, OH, OW, C, dtype=torch.bfloat16, device=gpu)
    layer(xd, y, residual=rd if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(xv, w, bn, stride=s, pad=1, groups=C, act=act, residual=rv if res_mode else None,
                          res_mode=res_mode)
    got = y.float().cpu().numpy()
    assert bf16_within_half_ulp(got, ref) <= 1.0
    assert rel_err(got, ref) <= TOL_BF16


@pytest.mark.parametrize("shape", [(2, 9, 13, 32, 1), (3, 14, 14, 48, 2), (1, 6, 131, 64, 2)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("act", [cb.ACT_RELU, cb.ACT_SILU])
def test_bf16_equals_fp32_kernel_rounded(gpu, shape, act):
    """Same fp32 arithmetic in both kernels: the bf16 output is the fp32 output rounded to
    nearest even, bit for bit."""
    N, H, W, C, s = shape
    x, w, bn, layer = _layer(shape, act, seed=11)
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(H, W)
    y16 = torch.empty(N, OH, OW, C, dtype=torch.bfloat16, device=gpu)
    y32 = torch.empty(N, OH, OW, C, device=gpu)
    layer(xd, y16)
    layer(torch.from_numpy(xv).to(gpu), y32)
    sync_check()
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))


def test_bf16_channel_slice_views_and_padded_rows(gpu, orc):
    """Input: channels [8, 8 + C) of a 96-channel bf16 buffer; output: channels [16, 16 + C) of a
    wider buffer with rows padded by 3 pixels.  Nothing outside the output view is written."""
    N, H, W, C, s = 2, 10, 12, 64, 1
    x, w, bn, layer = _layer((N, H, W, C, s), cb.ACT_SILU, seed=5)
    wide = np.random.default_rng(1).standard_normal((N, H, W, 96)).astype(np.float32)
    wide[..., 8:8 + C] = x
    wd, wv = to_dev_bf16(wide)
    xd, xv = wd[..., 8:8 + C], wv[..., 8:8 + C]
    buf = canary_buffer_bf16((N, H, W + 3, C + 32))
    y = buf[:, :, :W, 16:16 + C]
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(np.ascontiguousarray(xv), w, bn, stride=s, pad=1, groups=C, act=orc.ACT_SILU)
    assert bf16_within_half_ulp(y.float().cpu().numpy(), ref) <= 1.0
    assert is_canary_bf16(buf[:, :, W:, :]) and is_canary_bf16(buf[:, :, :W, :16])
    assert is_canary_bf16(buf[:, :, :W, 16 + C:])


@pytest.mark.parametrize("stride", [1, 2])
def test_bf16_depthwise_benchmark_layer_sampled(gpu, orc, stride):
    """The benchmark's layer ([64, 56, 56, 384]) with bf16 storage, on 8192 sampled outputs."""
    x, w, bn = synthetic.depthwise_layer()
    layer = ConvBnAct(w, bn, stride, 1, cb.ACT_RELU, groups=384)
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(56, 56)
    y = torch.empty(64, OH, OW, 384, dtype=torch.bfloat16, device=gpu)
    layer(xd, y)
    sync_check()
    idx = np.random.default_rng(stride).choice(y.numel(), 8192, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(xv, w, bn, idx, stride=stride, pad=1, groups=384, act=orc.ACT_RELU)
    got = y.reshape(-1)[torch.from_numpy(idx).to(gpu)].float().cpu().numpy()
    assert bf16_within_half_ulp(got, ref) <= 1.0
    assert bool(torch.isfinite(y.float()).all()) and float(y.float().min()) >= 0.0


def test_bf16_rejections(gpu):
    x, w, bn, layer = _layer((1, 6, 6, 12, 1), cb.ACT_RELU, seed=1)  # C % 8 != 0
    xd, _ = to_dev_bf16(x)
    with pytest.raises(cb.CbError) as e:
        layer(xd, torch.empty(1, 6, 6, 12, dtype=torch.bfloat16, device=gpu))
    assert e.value.status == cb.ERR_ALIGNMENT
    x, w, bn, layer = _layer((1, 6, 6, 16, 1), cb.ACT_RELU, seed=1)
    xd, _ = to_dev_bf16(x)
    with pytest.raises(cb.CbError) as e:  # mixed element types
        layer(xd, torch.empty(1, 6, 6, 16, device=gpu))
    assert e.value.status == cb.ERR_INVALID_ARG
    xs = torch.empty(1, 6, 6, 20, dtype=torch.bfloat16, device=gpu)[..., 2:18]  # 4-byte aligned pixels
    with pytest.raises(cb.CbError) as e:
        layer(xs, torch.empty(1, 6, 6, 16, dtype=torch.bfloat16, device=gpu))
    assert e.value.status == cb.ERR_ALIGNMENT
    xdense, wd, bnd = synthetic.dense_layer(12, 12, 8, N=1, k=3)  # 3x3 with 12 channels: no bf16 kernel
    dense = ConvBnAct(wd, bnd, 1, 1, cb.ACT_SILU)
    x16, _ = to_dev_bf16(xdense)
    y16 = torch.empty(1, 8, 8, 12, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(x16, y16, 3, 1, 1) == 0
    with pytest.raises(cb.CbError) as e:
        dense(x16, y16)
    assert e.value.status == cb.ERR_UNSUPPORTED
    with pytest.raises(TypeError):
        cb.conv_path(torch.empty(1, 8, 8, 32, dtype=torch.float16, device=gpu), y16, 3, 1, 1)
    sync_check()


PW_CASES = [
    # N, H, W, Ci, Co, act, res_mode
    (2, 9, 13, 16, 8, cb.ACT_SILU, 0), (2, 9, 13, 16, 16, cb.ACT_SILU, 2), (1, 5, 40, 32, 16, cb.ACT_RELU, 0),
    (2, 7, 7, 32, 32, cb.ACT_SILU, 2), (3, 4, 5, 8, 32, cb.ACT_RELU, 1), (1, 1, 1, 8, 4, cb.ACT_NONE, 0),
    (2, 33, 31, 16, 16, cb.ACT_SILU, 1),
]


@pytest.mark.parametrize("case", PW_CASES, ids=lambda c: "x".join(map(str, c)))
def test_bf16_pointwise(gpu, orc, case):
    N, H, W, Ci, Co, act, rm = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=1, seed=sum(case))
    layer = ConvBnAct(w, bn, 1, 0, act)
    xd, xv = to_dev_bf16(x)
    r = np.random.default_rng(4).standard_normal((N, H, W, Co)).astype(np.float32)
    rd, rv = to_dev_bf16(r)
    y = torch.empty(N, H, W, Co, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(xd, y, 1, 1, 0) == cb.PATH_POINTWISE
    layer(xd, y, residual=rd if rm else None, res_mode=rm)
    sync_check()
    ref = orc.conv_bn_act(xv, w, bn, stride=1, pad=0, act=act, residual=rv if rm else None, res_mode=rm)
    got = y.float().cpu().numpy()
    assert bf16_within_half_ulp(got, ref) <= 1.0
    assert rel_err(got, ref) <= TOL_BF16
    # the fp32 kernel runs the same sums: its output rounded to bf16 is this one, bit for bit
    y32 = torch.empty(N, H, W, Co, device=gpu)
    layer(torch.from_numpy(xv).to(gpu), y32, residual=torch.from_numpy(rv).to(gpu) if rm else None, res_mode=rm)
    sync_check()
    assert torch.equal(y.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))


def test_bf16_pointwise_in_place_residual_and_views(gpu, orc):
    """Residual added in place (r is y) and the output a channel slice of a wider bf16 buffer."""
    N, H, W, Ci, Co = 2, 6, 10, 16, 16
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=1, seed=21)
    layer = ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)
    xd, xv = to_dev_bf16(x)
    r = np.random.default_rng(6).standard_normal((N, H, W, Co)).astype(np.float32)
    rd, rv = to_dev_bf16(r)
    buf = canary_buffer_bf16((N, H, W, Co + 16))
    y = buf[..., 8:8 + Co]
    y.copy_(rd)
    layer(xd, y, residual=y, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = orc.conv_bn_act(xv, w, bn, stride=1, pad=0, act=orc.ACT_SILU, residual=rv, res_mode=orc.RES_POST_ACT)
    assert bf16_within_half_ulp(y.float().cpu().numpy(), ref) <= 1.0
    assert is_canary_bf16(buf[..., :8]) and is_canary_bf16(buf[..., 8 + Co:])


def test_bf16_pointwise_rejections(gpu):
    x, w, bn = synthetic.dense_layer(12, 32, 6, N=1, k=1, seed=2)  # 12 channels: no 16-byte bf16 rows
    layer = ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)
    xd, _ = to_dev_bf16(x)
    y = torch.empty(1, 6, 6, 32, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(xd, y, 1, 1, 0) == 0
    with pytest.raises(cb.CbError) as e:
        layer(xd, y)
    assert e.value.status == cb.ERR_UNSUPPORTED
    x, w, bn = synthetic.dense_layer(16, 16, 6, N=1, k=1, seed=3)
    layer = ConvBnAct(w, bn, 1, 0, cb.ACT_SILU)
    xs = torch.empty(1, 6, 6, 20, dtype=torch.bfloat16, device=gpu)[..., 2:18]  # 4-byte aligned pixels
    with pytest.raises(cb.CbError) as e:
        layer(xs, torch.empty(1, 6, 6, 16, dtype=torch.bfloat16, device=gpu))
    assert e.value.status == cb.ERR_ALIGNMENT
    sync_check()
