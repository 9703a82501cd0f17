"""GPU tests of the per-shape autotuner (cb_autotune_conv) and of every tile plan it can choose.

The tuner runs each candidate plan of a tensor-core layer on the caller's buffers and records the
fastest for the layer's shape.  The plans differ only in tiling, so every one must meet the TF32
bar against the fp64 oracle: the im2col tile widths are forced one by one here (the halo tile
shapes have their own forced tests); the tuned layer, and the layers launched after tuning, are
checked against the oracle; the table is keyed by shape and policy and can be cleared.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, TOL_TF32, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

TC_PATHS = (cb.PATH_TC_IM2COL, cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)


@pytest.fixture
def fresh_table():
    cb.autotune_clear()
    yield
    cb.autotune_clear()
    cb.set_kernel_policy(0)


@pytest.fixture
def igemm_force():
    cb.set_tuning("CB_IGEMM_FORCE", None)
    yield lambda v: cb.set_tuning("CB_IGEMM_FORCE", v)
    cb.set_tuning("CB_IGEMM_FORCE", None)


@pytest.mark.parametrize("bn", [16, 32, 48, 64, 96, 128, 192, 256])
def test_im2col_every_tile_width(gpu, orc, igemm_force, fresh_table, bn):
    """Stride 2, a ragged last pixel tile and a ragged last channel tile for each width (policy 2
    keeps the layer on the im2col-path kernel)."""
    igemm_force(f"{bn},0")
    cb.set_kernel_policy(2)
    N, H, Ci, Co = 2, 23, 32, 200
    x, w, bn_p = synthetic.dense_layer(Ci, Co, H, N=N, k=3, seed=bn)
    layer = ConvBnAct(w, bn_p, 2, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    y = torch.empty(N, OH, OW, Co, device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 2, 1) == cb.PATH_TC_IM2COL
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn_p, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("case", [
    # N, H, Cin, Cout, stride: halo-eligible, stride-2 im2col, narrow 1x1-free 3x3
    (2, 20, 64, 96, 1), (1, 40, 128, 128, 1), (2, 21, 32, 64, 2), (1, 16, 16, 48, 1),
], ids=lambda c: "x".join(map(str, c)))
def test_autotune_result_and_later_calls(gpu, orc, fresh_table, case):
    N, H, Ci, Co, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=N, k=3, seed=sum(case))
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    xd = to_dev(x)
    y0 = torch.empty(N, OH, OW, Co, device="cuda")
    assert cb.conv_path(xd, y0, 3, s, 1) in TC_PATHS
    layer.autotune(xd, y0)
    sync_check()
    assert cb.autotune_entries() == 1
    assert cb.conv_path(xd, y0, 3, s, 1) in TC_PATHS
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, act=orc.ACT_SILU)
    assert rel_err(y0.cpu().numpy(), ref) <= TOL_TF32
    y1 = torch.full_like(y0, float("nan"))
    layer(xd, y1)  # the recorded plan
    sync_check()
    assert torch.equal(y0, y1)  # same plan, same summation order


def test_autotune_with_residual_and_slice_views(gpu, orc, fresh_table):
    """The tuner times the caller's epilogue and views; the in-place residual is applied once."""
    N, H, W, Ci, Co = 2, 12, 30, 64, 64
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=5)
    r = np.random.default_rng(9).standard_normal((N, H, W, Co)).astype(np.float32)
    layer = ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)
    xd = to_dev(x)
    rd = to_dev(r)
    buf = torch.zeros(N, H, W, Co + 32, device="cuda")
    y = buf[..., 16:16 + Co]
    layer.autotune(xd, y, residual=rd, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU, residual=r, res_mode=orc.RES_POST_ACT)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert float(buf[..., :16].abs().max()) == 0.0 and float(buf[..., 16 + Co:].abs().max()) == 0.0


def test_autotune_single_kernel_layers_record_nothing(gpu, orc, fresh_table):
    """Depthwise and other CUDA-core layers have one kernel: launched once, nothing recorded."""
    x, w, bn = synthetic.dense_layer(3, 16, 24, N=1, k=3, seed=2)  # stem: the stem kernel
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(24, 24)
    y = torch.empty(1, OH, OW, 16, device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 2, 1) == cb.PATH_STEM
    layer.autotune(xd, y)
    sync_check()
    assert cb.autotune_entries() == 0
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32

    rng = np.random.default_rng(3)
    xdw = rng.standard_normal((2, 10, 10, 64)).astype(np.float32)
    wdw = rng.standard_normal((64, 1, 3, 3)).astype(np.float32) * 0.3
    bndw = synthetic.bn_params(rng, 64)
    dw = ConvBnAct(wdw, bndw, 1, 1, cb.ACT_RELU, groups=64)
    ydw = torch.empty(2, 10, 10, 64, device="cuda")
    dw.autotune(to_dev(xdw), ydw)
    sync_check()
    assert cb.autotune_entries() == 0
    ref = orc.conv_bn_act(xdw, wdw, bndw, stride=1, pad=1, groups=64, act=orc.ACT_RELU)
    assert rel_err(ydw.cpu().numpy(), ref) <= TOL_FP32


def test_autotune_keyed_by_shape_and_policy(gpu, fresh_table):
    x, w, bn = synthetic.dense_layer(64, 64, 16, N=1, k=3, seed=8)
    layer = ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)
    xd = to_dev(x)
    y = torch.empty(1, 16, 16, 64, device="cuda")
    layer.autotune(xd, y)
    sync_check()
    assert cb.autotune_entries() == 1
    layer.autotune(xd, y)  # re-tuning the same shape replaces its entry
    assert cb.autotune_entries() == 1
    cb.set_kernel_policy(2)  # another policy: its own key; the halo kernels are off
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_TC_IM2COL
    layer.autotune(xd, y)
    sync_check()
    assert cb.autotune_entries() == 2
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_TC_IM2COL
    cb.set_kernel_policy(1)  # CUDA-core only: a tuned tensor-core plan never applies
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_DIRECT
    cb.set_kernel_policy(0)
    cb.autotune_clear()
    assert cb.autotune_entries() == 0
