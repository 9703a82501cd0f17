"""GPU parity of the bf16 storage variant on the tensor cores: dense 3x3 and 1x1 conv + folded BN +
activation (+ residual) with x, y, the residual and the weights held as bfloat16 and the products
summed in fp32 (tcgen05 kind::f16 MMAs), in both tensor-core kernels (halo tiles and im2col).

Two oracle references, both fp64 on the bf16 input values:
  * with the bf16 weights the kernel multiplies (cb_convert_weights_bf16's output): the products
    are exact, so every output must lie within half a bf16 unit in the last place of the oracle
    (2^-8 of the value) plus the fp32 accumulation bar -- the kernel adds nothing but fp32 sums
    and the final rounding;
  * with the original fp32 weights: within 5e-3 of max|oracle| (the bf16 storage bar).
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_BF16, bf16_within_half_ulp, canary_buffer_bf16, is_canary_bf16, rel_err, sync_check, \
    to_dev_bf16

pytestmark = pytest.mark.gpu

TC_PATHS = (cb.PATH_TC_IM2COL, cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)

CASES = [
    # N, H, W, Cin, Cout, k, stride: halo tiles of 128-, 64- and 32-byte rows, stride-2 phase tiles,
    # ragged channel tiles, images narrower and wider than a tile row, 1x1 layers (im2col kernel)
    (2, 10, 12, 16, 32, 3, 1), (1, 17, 9, 32, 16, 3, 2), (2, 9, 7, 64, 64, 3, 1), (1, 20, 20, 128, 256, 3, 2),
    (1, 40, 40, 64, 128, 3, 2), (2, 7, 7, 192, 192, 3, 1), (1, 5, 80, 96, 100, 3, 1), (2, 11, 13, 48, 40, 3, 1),
    (2, 14, 14, 48, 96, 1, 2), (3, 8, 8, 64, 64, 1, 1), (2, 9, 7, 48, 8, 1, 1), (1, 6, 6, 256, 384, 1, 1),
    (1, 16, 16, 16, 48, 3, 2), (1, 1, 1, 32, 32, 3, 1),
]


def _run(case, act=cb.ACT_SILU, seed=0, residual=None, res_mode=0, y=None):
    N, H, W, Ci, Co, k, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=k, seed=seed)
    layer = ConvBnAct(w, bn, s, k // 2, act, dtype=torch.bfloat16)
    assert layer.tc_weights
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(H, W)
    if y is None:
        y = torch.empty(N, OH, OW, Co, dtype=torch.bfloat16, device="cuda")
    assert cb.conv_path(xd, y, k, s, k // 2) in TC_PATHS
    layer(xd, y, residual=residual, res_mode=res_mode)
    sync_check()
    # the weights as the kernel holds them (rounded to bf16 by the library), back in OIHW order
    wb = cb.convert_weights_bf16(w).float().numpy()
    return x, xv, w, wb, bn, y


def _check(orc, xv, w, wb, bn, got, s, pad, act=cb.ACT_SILU, r=None, res_mode=0):
    kw = dict(stride=s, pad=pad, act=act, residual=r, res_mode=res_mode)
    ref_b = orc.conv_bn_act(xv, wb, bn, **kw)
    assert bf16_within_half_ulp(got, ref_b) <= 1.0
    assert rel_err(got, orc.conv_bn_act(xv, w, bn, **kw)) <= TOL_BF16


@pytest.fixture(params=[0, 2], ids=["auto", "im2col"])
def policy(request, gpu):
    cb.set_kernel_policy(request.param)
    yield request.param
    cb.set_kernel_policy(0)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_bf16_tc_silu(gpu, orc, policy, case):
    N, H, W, Ci, Co, k, s = case
    x, xv, w, wb, bn, y = _run(case, seed=sum(case))
    _check(orc, xv, w, wb, bn, y.float().cpu().numpy(), s, k // 2)


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 1), (2, 2), (0, 2), (1, 0)])
def test_bf16_tc_epilogue_variants(gpu, orc, act, res_mode):
    case = (2, 9, 10, 64, 48, 3, 1)
    N, H, W, Ci, Co, k, s = case
    r = np.random.default_rng(act + 5 * res_mode).standard_normal((N, H, W, Co)).astype(np.float32)
    rd, rv = to_dev_bf16(r)
    x, xv, w, wb, bn, y = _run(case, act=act, seed=act + 7 * res_mode, residual=rd if res_mode else None,
                               res_mode=res_mode)
    _check(orc, xv, w, wb, bn, y.float().cpu().numpy(), s, 1, act=act, r=rv if res_mode else None,
           res_mode=res_mode)


@pytest.mark.parametrize("force", ["cm", "cm192", "32", "64", "128", "256", "64,0,0,0,2", "128,0,2", "cm,0,2",
                                   "cm192,0,2"])
def test_bf16_halo_every_tile(gpu, orc, force):
    """Every halo tile shape (forced), incl. split K over CTA pairs and sub-tiles, in bf16."""
    case = (2, 20, 20, 128, 128, 3, 1)
    with cb.tuning("CB_HALO_FORCE", force):
        x, xv, w, wb, bn, y = _run(case, seed=len(force))
        assert cb.conv_path(to_dev_bf16(x)[0], y, 3, 1, 1) in (cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)
    _check(orc, xv, w, wb, bn, y.float().cpu().numpy(), 1, 1)


def test_bf16_tc_output_view_and_in_place_residual(gpu, orc):
    """Output a channel slice of a wider bf16 buffer with padded rows, the residual added in place;
    the bytes around the slice keep their canaries."""
    N, H, W, Ci, Co = 2, 12, 18, 32, 64
    r = np.random.default_rng(8).standard_normal((N, H, W, Co)).astype(np.float32)
    rd, rv = to_dev_bf16(r)
    buf = canary_buffer_bf16((N, H, W + 3, Co + 16))
    y = buf[:, :, :W, 8:8 + Co]
    y.copy_(rd)
    x, xv, w, wb, bn, y = _run((N, H, W, Ci, Co, 3, 1), seed=8, residual=y, res_mode=cb.RES_POST_ACT, y=y)
    _check(orc, xv, w, wb, bn, y.float().cpu().numpy(), 1, 1, r=rv, res_mode=cb.RES_POST_ACT)
    assert is_canary_bf16(buf[..., :8]) and is_canary_bf16(buf[..., 8 + Co:]) and is_canary_bf16(buf[:, :, W:])


def test_bf16_tc_autotune(gpu, orc):
    """The tuner times bf16 plans separately from fp32 ones (the table is keyed by element type)."""
    cb.autotune_clear()
    try:
        case = (2, 20, 20, 64, 64, 3, 1)
        N, H, W, Ci, Co, k, s = case
        x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=k, seed=4)
        layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU, dtype=torch.bfloat16)
        xd, xv = to_dev_bf16(x)
        y = torch.empty(N, H, W, Co, dtype=torch.bfloat16, device=gpu)
        layer.autotune(xd, y)
        assert cb.autotune_entries() == 1
        y.fill_(float("nan"))
        layer(xd, y)
        sync_check()
        _check(orc, xv, w, cb.convert_weights_bf16(w).float().numpy(), bn, y.float().cpu().numpy(), 1, 1)
    finally:
        cb.autotune_clear()


@pytest.mark.parametrize("layer_spec", synthetic.DENSE_SWEEP[1:], ids=lambda s: "%d-%d@%d_s%d" % s)
def test_bf16_dense_sweep_batch16_full(gpu, orc, layer_spec):
    """The tensor-core layers of the dense sweep at batch 16 in bf16, every output checked."""
    ci, co, H, s = layer_spec
    x, w, bn = synthetic.dense_layer(ci, co, H, N=16, k=3)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU, dtype=torch.bfloat16)
    xd, xv = to_dev_bf16(x)
    OH, OW = layer.out_hw(H, H)
    y = torch.empty(16, OH, OW, co, dtype=torch.bfloat16, device=gpu)
    layer(xd, y)
    sync_check()
    _check(orc, xv, w, cb.convert_weights_bf16(w).float().numpy(), bn, y.float().cpu().numpy(), s, 1)
