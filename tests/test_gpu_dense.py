"""GPU parity: dense 1x1 / 3x3 conv + folded BN + activation (+ residual) vs the fp64 oracle.

Layers with Cin % 4 == 0 and Cin >= 8 (1x1) or >= 16 (3x3) run on the tcgen05 implicit GEMM (TF32
inputs, fp32 accumulate): bar 5e-3 relative to max.  Everything else (and
every layer under kernel policy 1) runs on the fp32 direct kernel: bar 1e-5.
Policy 2 keeps the tensor cores but replaces the halo-tile kernel with the
im2col one, so both tensor-core kernels see every shape here.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, TOL_TF32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

DENSE = [
    # N, H, W, Cin, Cout, k, stride
    (2, 10, 12, 16, 32, 3, 1), (1, 17, 9, 32, 16, 3, 2), (3, 8, 8, 64, 64, 1, 1), (2, 9, 7, 48, 8, 1, 1),
    (1, 20, 20, 128, 256, 3, 2), (1, 40, 40, 64, 128, 3, 2), (2, 7, 7, 192, 192, 1, 1), (1, 6, 6, 256, 384, 1, 1),
    (1, 5, 5, 96, 96, 3, 1), (2, 13, 11, 16, 48, 3, 1), (1, 3, 3, 20, 24, 3, 1), (2, 14, 14, 48, 96, 1, 2),
    (1, 1, 1, 16, 16, 3, 1), (1, 30, 30, 36, 40, 3, 1),
    (2, 17, 13, 8, 8, 3, 1), (2, 16, 16, 8, 16, 3, 2), (2, 11, 9, 16, 8, 1, 1), (1, 12, 12, 12, 20, 3, 1),
    (2, 10, 10, 4, 16, 3, 1), (1, 9, 9, 24, 32, 1, 2), (1, 40, 40, 16, 16, 1, 1),
    (2, 9, 11, 8, 24, 1, 1), (1, 7, 9, 12, 16, 1, 1), (2, 33, 35, 3, 16, 3, 2), (1, 21, 19, 16, 40, 3, 1),
    # 8 -> <= 8 channel 3x3 stride 1 (four output rows per thread): ragged tile rows and columns
    (1, 37, 70, 8, 8, 3, 1), (2, 9, 33, 8, 4, 3, 1),
]


def _is_tc(cin, cout, k=3, stride=1):
    return cb.layer_uses_tensor_cores(cin, cout, k, stride)


@pytest.fixture(params=[0, 1, 2], ids=["auto", "direct", "im2col"])
def policy(request, gpu):
    cb.set_kernel_policy(request.param)
    yield request.param
    cb.set_kernel_policy(0)


@pytest.mark.parametrize("case", DENSE, ids=lambda s: "x".join(map(str, s)))
def test_dense_silu(gpu, policy, orc, case):
    N, H, W, Ci, Co, k, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=k, seed=hash(case) % 1000)
    pad = k // 2
    layer = ConvBnAct(w, bn, s, pad, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, W)
    y = torch.empty(N, OH, OW, Co, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=pad, act=orc.ACT_SILU)
    tol = TOL_TF32 if _is_tc(Ci, Co, k, s) else TOL_FP32
    assert rel_err(y.cpu().numpy(), ref) <= tol


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 0), (1, 1), (2, 2), (0, 2)])
@pytest.mark.parametrize("k", [1, 3])
def test_dense_epilogue_variants(gpu, policy, orc, act, res_mode, k):
    N, H, W, Ci, Co = 2, 9, 10, 32, 48
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=k, seed=act + 5 * res_mode)
    r = np.random.default_rng(4).standard_normal((N, H, W, Co)).astype(np.float32)
    layer = ConvBnAct(w, bn, 1, k // 2, act)
    y = torch.empty(N, H, W, Co, device=gpu)
    layer(to_dev(x), y, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=k // 2, act=act, residual=r if res_mode else None,
                          res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= (TOL_TF32 if _is_tc(Ci, Co, k) else TOL_FP32)


@pytest.mark.parametrize("stem", [(1, 48, 28, 1), (3, 16, 64, 2), (3, 16, 33, 2), (8, 8, 20, 1)])
def test_small_channel_direct(gpu, orc, stem):
    Ci, Co, H, s = stem
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=2, k=3, seed=Ci * Co + H)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    y = torch.empty(2, OH, OW, Co, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    tol = TOL_TF32 if _is_tc(Ci, Co, 3, s) else TOL_FP32  # 8-channel stride-1 layers take halo tiles
    assert rel_err(y.cpu().numpy(), orc.conv_bn_act(x, w, bn, stride=s, pad=1, act=orc.ACT_SILU)) <= tol


def test_nchw_input_stem(gpu, orc):
    """The stem reads a planar [N, 3, H, W] tensor (the preprocess output) directly."""
    x, w, bn = synthetic.dense_layer(3, 16, 48, 64, N=2, k=3, seed=5)
    xp = np.ascontiguousarray(x.transpose(0, 3, 1, 2))
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    y = torch.empty(2, 24, 32, 16, device=gpu)
    layer(to_dev(xp), y, x_layout=cb.LAYOUT_NCHW)
    sync_check()
    ref = orc.conv_bn_act(xp, w, bn, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("ow_case", [(80, 40, 64), (40, 20, 128)], ids=["OW40", "OW20"])
def test_padded_output_rows_not_overwritten(gpu, policy, orc, ow_case):
    """Rows padded to a multiple of 16 columns: the masked epilogue leaves the padding alone
    (the OW=40 / OW=20 overflow case of the TMA-store bug)."""
    H, OW, C = ow_case
    x, w, bn = synthetic.dense_layer(C, C, H, N=1, k=3, seed=H)
    pad_w = (OW + 15) // 16 * 16
    ybuf = canary_buffer((1, OW, pad_w, 2 * C))
    y = ybuf[:, :, :OW, :C]
    ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)(to_dev(x), y)
    sync_check()
    assert is_canary(ybuf[:, :, OW:, :]) and is_canary(ybuf[:, :, :OW, C:])
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= (TOL_TF32 if policy != 1 else TOL_FP32)


@pytest.mark.parametrize("case", synthetic.DENSE_SWEEP, ids=lambda s: "%d-%d@%d_s%d" % s)
def test_dense_sweep_batch1_full(gpu, orc, case):
    """The dense 3x3 sweep at batch 1, every output checked."""
    Ci, Co, H, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=1, k=3)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    y = torch.empty(1, OH, OW, Co, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= (TOL_TF32 if _is_tc(Ci, Co, 3, s) else TOL_FP32)


@pytest.mark.parametrize("case", synthetic.DENSE_SWEEP, ids=lambda s: "%d-%d@%d_s%d" % s)
def test_dense_sweep_batch16_sampled(gpu, orc, case):
    Ci, Co, H, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=16, k=3)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    y = torch.empty(16, OH, OW, Co, device=gpu)
    layer(to_dev(x), y)
    sync_check()
    idx = np.random.default_rng(Ci).choice(y.numel(), min(y.numel(), 6000), replace=False)
    idx = np.concatenate([idx, [y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=s, pad=1, act=orc.ACT_SILU)
    got = y.reshape(-1)[torch.from_numpy(idx).to(gpu)].cpu().numpy()
    assert rel_err(got, ref) <= (TOL_TF32 if _is_tc(Ci, Co, 3, s) else TOL_FP32)
