"""GPU parity: depthwise 3x3 + folded BN + activation (+ residual) vs the fp64 oracle.

Both depthwise kernels are exercised: the TMA-fed persistent kernel (policy 0)
and the plain CUDA-core kernel (policy 1).  Bar: max|gpu - oracle| / max|oracle|
<= 1e-5 (fp32 CUDA-core arithmetic).
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [
    # N, H, W, C, stride
    (2, 9, 13, 32, 1), (2, 9, 13, 32, 2), (3, 14, 14, 48, 2), (2, 7, 7, 192, 1),
    (1, 20, 20, 12, 1), (1, 5, 130, 64, 1), (1, 6, 131, 64, 2), (1, 1, 1, 4, 1), (2, 3, 3, 6, 1),
    (1, 2, 2, 8, 2), (4, 28, 28, 48, 2), (2, 14, 14, 96, 1), (1, 33, 17, 36, 1),
]


@pytest.fixture(params=[0, 1], ids=["tma", "simple"])
def policy(request, gpu):
    cb.set_kernel_policy(request.param)
    yield request.param
    cb.set_kernel_policy(0)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_depthwise_relu(gpu, policy, orc, shape):
    N, H, W, C, s = shape
    x, w, bn = synthetic.depthwise_layer(N, C, H, W, seed=hash(shape) % 10000)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_RELU, groups=C)
    OH, OW = layer.out_hw(H, W)
    y = torch.empty(N, OH, OW, C, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, groups=C, act=orc.ACT_RELU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("act,res_mode", [(0, 0), (2, 0), (1, 1), (2, 2), (0, 1)])
def test_depthwise_epilogue_variants(gpu, policy, orc, act, res_mode):
    N, H, W, C, s = 2, 11, 9, 64, 1
    x, w, bn = synthetic.depthwise_layer(N, C, H, W, seed=7 + act + 3 * res_mode)
    r = np.random.default_rng(3).standard_normal((N, H, W, C)).astype(np.float32)
    layer = ConvBnAct(w, bn, s, 1, act, groups=C)
    y = torch.empty(N, H, W, C, device=gpu)
    layer(to_dev(x), y, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, groups=C, act=act, residual=r if res_mode else None,
                          res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_depthwise_channel_slice_views_and_padded_rows(gpu, policy, orc):
    """Input is a channel slice of a wider buffer; output rows are padded to a multiple of 16
    columns and the padding (canary) must stay untouched."""
    N, H, W, C = 2, 40, 40, 32
    x, w, bn = synthetic.depthwise_layer(N, C, H, W, seed=11)
    wide = torch.zeros(N, H, W, C + 16, device=gpu)
    wide[..., 8:8 + C] = to_dev(x)
    for s, OW in ((1, 40), (2, 20)):
        pad_w = (OW + 15) // 16 * 16
        ybuf = canary_buffer((N, OW, pad_w, C))  # OH == OW here
        y = ybuf[:, :, :OW, :]
        layer = ConvBnAct(w, bn, s, 1, cb.ACT_RELU, groups=C)
        layer(wide[..., 8:8 + C], y)
        sync_check()
        assert is_canary(ybuf[:, :, OW:, :]), "padding columns were written"
        ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, groups=C, act=orc.ACT_RELU)
        assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("stride", [1, 2])
def test_depthwise_full_workload_sampled(gpu, orc, stride):
    """The benchmark's layer ([64, 56, 56, 384], default kernel choice) checked on 8192 sampled outputs."""
    x, w, bn = synthetic.depthwise_layer()
    layer = ConvBnAct(w, bn, stride, 1, cb.ACT_RELU, groups=384)
    OH, OW = layer.out_hw(56, 56)
    y = torch.empty(64, OH, OW, 384, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    idx = np.random.default_rng(stride).choice(y.numel(), 8192, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=stride, pad=1, groups=384, act=orc.ACT_RELU)
    got = y.reshape(-1)[torch.from_numpy(idx).to(gpu)].cpu().numpy()
    assert rel_err(got, ref) <= TOL_FP32
    # a property that holds everywhere: ReLU output is non-negative and finite
    assert bool(torch.isfinite(y).all()) and float(y.min()) >= 0.0


def test_depthwise_empty_batch(gpu):
    x, w, bn = synthetic.depthwise_layer(1, 8, 5, 5)
    layer = ConvBnAct(w, bn, 1, 1, cb.ACT_RELU, groups=8)
    y = torch.empty(0, 5, 5, 8, device=gpu)
    layer(torch.empty(0, 5, 5, 8, device=gpu), y)
    sync_check()
