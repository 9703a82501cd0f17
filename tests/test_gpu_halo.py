"""GPU parity of the halo-tile tensor-core kernel (3x3, stride 1, pad 1, Cin % 32 == 0), in both of
its tile shapes: pixel-major (128 pixels x up to 256 channels) and channel-major (256 or 192 pixels x
128 channels, the channels as the MMA's M).

Each output is checked against the fp64 oracle at the TF32 bar (5e-3 of max|oracle|).  The
shapes cover one and several tiles per image, tiles that wrap across output rows, images narrower
than a tile row and wider than one, channel counts that leave a ragged last channel tile, every
tile width the kernel has (forced through CB_HALO_FORCE), the epilogue variants, channel-slice
output views with padded rows (canaries must survive) and the in-place residual.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_TF32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

CASES = [
    # N, H, W, Cin, Cout
    (1, 1, 1, 32, 32), (2, 3, 5, 32, 16), (1, 20, 20, 64, 64), (2, 7, 40, 32, 40),
    (1, 5, 80, 96, 128), (1, 4, 126, 32, 32), (1, 6, 150, 32, 32), (3, 9, 13, 64, 100),
    (1, 20, 20, 256, 256), (2, 11, 17, 128, 384), (1, 40, 40, 128, 128), (1, 2, 2, 32, 8),
]


@pytest.fixture
def halo_force():
    cb.set_tuning("CB_HALO_FORCE", None)
    yield lambda v: cb.set_tuning("CB_HALO_FORCE", v)
    cb.set_tuning("CB_HALO_FORCE", None)


def _run(x, w, bn, act=cb.ACT_SILU, residual=None, res_mode=0, y=None):
    N, H, W, _ = x.shape
    layer = ConvBnAct(w, bn, 1, 1, act)
    if y is None:
        y = torch.empty(N, H, W, w.shape[0], device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) in (cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)
    layer(xd, y, residual=residual, res_mode=res_mode)
    sync_check()
    return y


@pytest.mark.parametrize("case", CASES, ids=lambda s: "x".join(map(str, s)))
def test_halo_silu(gpu, orc, case):
    N, H, W, Ci, Co = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case))
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("bn_force", ["32,0", "64,0", "128,0", "256,0", "128,3", "64,16", "cm", "cm,2", "cm192",
                                      "cm192,2",
                                      # taps per weight-ring stage (one copy each): 9, 3 and 1
                                      "32,0,1,9", "64,0,1,3", "128,0,1,3", "128,0,1,1", "cm,0,1,3", "cm,0,1,1",
                                      "cm192,0,1,3", "cm192,0,1,1", "256,0,1,1"])
def test_halo_tile_widths(gpu, orc, halo_force, bn_force):
    halo_force(bn_force)
    x, w, bn = synthetic.dense_layer(64, 200, 10, 23, N=2, k=3, seed=3)
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 0), (1, 1), (2, 2), (0, 2), (2, 1)])
def test_halo_epilogue_variants(gpu, orc, act, res_mode):
    N, H, W, Ci, Co = 2, 9, 30, 32, 48
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=act + 5 * res_mode)
    r = np.random.default_rng(4).standard_normal((N, H, W, Co)).astype(np.float32)
    y = _run(x, w, bn, act=act, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r if res_mode else None,
                          res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


def test_halo_channel_slice_views_padded_rows(gpu, orc):
    """Output into channels [36, 36+Co) of a wider buffer whose rows are padded: every element
    outside the view keeps its canary."""
    N, H, W, Ci, Co = 2, 13, 21, 64, 40
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=11)
    buf = canary_buffer((N, H, W + 3, 36 + Co + 20))
    y = buf[:, :, :W, 36:36 + Co]
    _run(x, w, bn, y=y)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, W:, :]) and is_canary(buf[:, :, :W, :36]) and is_canary(buf[:, :, :W, 36 + Co:])


def test_halo_inplace_residual(gpu, orc):
    N, H, W, C = 1, 16, 24, 64
    x, w, bn = synthetic.dense_layer(C, C, H, W, N=N, k=3, seed=12)
    r = np.random.default_rng(5).standard_normal((N, H, W, C)).astype(np.float32)
    y = to_dev(r)
    _run(x, w, bn, residual=y, res_mode=cb.RES_POST_ACT, y=y)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU, residual=r, res_mode=orc.RES_POST_ACT)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


def test_halo_matches_im2col_kernel(gpu):
    """The two tensor-core kernels compute the same TF32 products in a different order; both
    round their outputs to TF32 (10 stored mantissa bits), so a different fp32 sum may flip the
    last stored bit: 2^-10 of a value at most."""
    x, w, bn = synthetic.dense_layer(128, 128, 40, N=2, k=3, seed=13)
    y0 = _run(x, w, bn)
    cb.set_kernel_policy(2)
    try:
        layer = ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)
        y1 = torch.empty_like(y0)
        xd = to_dev(x)
        assert cb.conv_path(xd, y1, 3, 1, 1) == cb.PATH_TC_IM2COL
        layer(xd, y1)
        sync_check()
    finally:
        cb.set_kernel_policy(0)
    assert rel_err(y0.cpu().numpy(), y1.cpu().numpy()) <= 2.0 ** -10


def test_halo_not_taken_outside_its_shapes(gpu):
    x = torch.empty(1, 8, 8, 36, device="cuda")  # Cin % 8 != 0
    y = torch.empty(1, 8, 8, 32, device="cuda")
    assert cb.conv_path(x, y, 3, 1, 1) == cb.PATH_TC_IM2COL
    x = torch.empty(1, 8, 8, 40, device="cuda")  # stride 2 with Cin % 16 != 0
    y = torch.empty(1, 4, 4, 32, device="cuda")
    assert cb.conv_path(x, y, 3, 2, 1) == cb.PATH_TC_IM2COL
    x = torch.empty(1, 8, 8, 32, device="cuda")  # 1x1
    y = torch.empty(1, 8, 8, 48, device="cuda")
    assert cb.conv_path(x, y, 1, 1, 0) == cb.PATH_TC_IM2COL


@pytest.mark.parametrize("case", [(64, 64, 80), (128, 128, 40), (256, 256, 20)], ids=lambda s: "%d-%d@%d" % s)
def test_halo_dense_sweep_batch16_sampled(gpu, orc, case):
    """The stride-1 layers of the dense sweep at batch 16, in the launch configuration the
    benchmark times; sampled outputs against the oracle point by point."""
    Ci, Co, H = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=16, k=3)
    y = _run(x, w, bn)
    idx = np.random.default_rng(Ci).choice(y.numel(), 6000, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=1, pad=1, act=orc.ACT_SILU)
    got = y.reshape(-1)[torch.from_numpy(idx).to("cuda")].cpu().numpy()
    assert rel_err(got, ref) <= TOL_TF32


CM_CASES = [
    # N, H, W, Cin, Cout: one and several 256-pixel tiles, ragged channel tiles, tiny images
    (1, 1, 1, 32, 128), (2, 3, 5, 32, 128), (1, 20, 20, 128, 128), (2, 9, 40, 64, 200),
    (1, 16, 16, 256, 256), (3, 7, 13, 32, 100), (1, 5, 60, 96, 384),
]


@pytest.mark.parametrize("px", [256, 192])
@pytest.mark.parametrize("case", CM_CASES, ids=lambda s: "x".join(map(str, s)))
def test_halo_channel_major(gpu, orc, halo_force, case, px):
    halo_force(f"cm{px}")
    N, H, W, Ci, Co = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case) + 7)
    layer = ConvBnAct(w, bn, 1, 1, cb.ACT_SILU)
    y = torch.empty(N, H, W, Co, device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_TC_HALO_CM
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("px", [256, 192])
@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2), (0, 0)])
def test_halo_channel_major_epilogues_and_views(gpu, orc, halo_force, act, res_mode, px):
    """Channel-major tiles into a channel slice of a padded buffer, with a residual."""
    halo_force(f"cm{px}")
    N, H, W, Ci, Co = 2, 11, 19, 64, 128
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=31 + act)
    r = np.random.default_rng(6).standard_normal((N, H, W, Co)).astype(np.float32)
    buf = canary_buffer((N, H, W + 5, Co + 36))
    y = buf[:, :, :W, 32:32 + Co]
    layer = ConvBnAct(w, bn, 1, 1, act)
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_TC_HALO_CM
    layer(xd, y, residual=to_dev(r) if res_mode else None, res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, W:, :]) and is_canary(buf[:, :, :W, :32]) and is_canary(buf[:, :, :W, 32 + Co:])


SPLIT_CASES = [
    # N, H, W, Cin, Cout, CB_HALO_FORCE: one tile per CTA pair, K chunks split between the pair
    (1, 20, 20, 128, 256, "256,0,2"), (1, 9, 13, 96, 128, "128,0,2"), (2, 5, 7, 64, 64, "64,0,2"),
    (1, 20, 20, 256, 256, "cm,0,2"), (1, 11, 17, 96, 200, "cm,0,2"), (2, 12, 12, 64, 100, "128,0,2"),
    (1, 20, 20, 256, 256, "cm192,0,2"), (1, 11, 17, 96, 200, "cm192,0,2"), (1, 13, 15, 64, 128, "cm192,0,2"),
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda s: "x".join(map(str, s[:5])) + "-" + s[5])
def test_halo_split_k(gpu, orc, halo_force, case):
    """Clusters of two CTAs sharing each tile's channel chunks (odd chunk counts included) and
    exchanging half accumulators through distributed shared memory."""
    N, H, W, Ci, Co, force = case
    halo_force(force)
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case[:5]))
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("force", ["128,0,2", "cm,0,2", "cm192,0,2"])
@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2)])
def test_halo_split_k_epilogues_and_views(gpu, orc, halo_force, force, act, res_mode):
    """Split-K tiles into a channel slice of a padded buffer, with a residual: nothing outside
    the view is written."""
    halo_force(force)
    N, H, W, Ci, Co = 1, 10, 18, 64, 128
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=41 + act)
    r = np.random.default_rng(7).standard_normal((N, H, W, Co)).astype(np.float32)
    buf = canary_buffer((N, H, W + 3, Co + 40))
    y = buf[:, :, :W, 8:8 + Co]
    layer = ConvBnAct(w, bn, 1, 1, act)
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) in (cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)
    layer(xd, y, residual=to_dev(r), res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, W:, :]) and is_canary(buf[:, :, :W, :8]) and is_canary(buf[:, :, :W, 8 + Co:])


KC16_CASES = [
    # N, H, W, Cin, Cout: 16-channel chunks (Cin % 32 == 16), pixel-major 128 x {32, 64} tiles
    (2, 7, 40, 16, 32), (1, 20, 20, 48, 64), (2, 9, 13, 16, 16), (1, 5, 80, 80, 64), (3, 11, 17, 16, 40),
    (1, 1, 1, 16, 32),
]


@pytest.mark.parametrize("case", KC16_CASES, ids=lambda s: "x".join(map(str, s)))
def test_halo_16_channel_chunks(gpu, orc, case):
    """64-byte pixel rows with the 64-byte swizzle: the nine taps start their descriptors at any
    64-byte row of the halo tile."""
    N, H, W, Ci, Co = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case) + 3)
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("force", ["32,0,1,9", "64,0,1,3", "64,0,1,1"])
@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2)])
def test_halo_16_channel_chunks_epilogues_and_views(gpu, orc, halo_force, force, act, res_mode):
    halo_force(force)
    N, H, W, Ci, Co = 2, 10, 33, 48, 64
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=61 + act)
    r = np.random.default_rng(8).standard_normal((N, H, W, Co)).astype(np.float32)
    buf = canary_buffer((N, H, W + 2, Co + 16))
    y = buf[:, :, :W, 4:4 + Co]
    layer = ConvBnAct(w, bn, 1, 1, act)
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, 1, 1) == cb.PATH_TC_HALO
    layer(xd, y, residual=to_dev(r), res_mode=res_mode)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, W:, :]) and is_canary(buf[:, :, :W, :4]) and is_canary(buf[:, :, :W, 4 + Co:])


def _run_s(x, w, bn, s, act=cb.ACT_SILU, residual=None, res_mode=0, y=None):
    N, H, W, _ = x.shape
    layer = ConvBnAct(w, bn, s, 1, act)
    OH, OW = layer.out_hw(H, W)
    if y is None:
        y = torch.empty(N, OH, OW, w.shape[0], device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, 3, s, 1) in (cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)
    layer(xd, y, residual=residual, res_mode=res_mode)
    sync_check()
    return y


S2_CASES = [
    # N, H, W, Cin, Cout: stride 2 as four phase tiles per 16-channel chunk; one and several
    # column blocks, odd sizes, tiny images, 128 output channels
    (2, 32, 32, 16, 32), (1, 40, 40, 16, 64), (2, 21, 23, 32, 64), (1, 9, 13, 48, 128), (1, 30, 300, 16, 32),
    (1, 2, 5, 16, 32), (3, 17, 33, 64, 100), (1, 1, 1, 16, 16),
]


@pytest.mark.parametrize("case", S2_CASES, ids=lambda s: "x".join(map(str, s)))
def test_halo_stride2_phases(gpu, orc, case):
    N, H, W, Ci, Co = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case) + 11)
    y = _run_s(x, w, bn, 2)
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2), (0, 0)])
def test_halo_stride2_epilogues_and_views(gpu, orc, act, res_mode):
    N, H, W, Ci, Co = 2, 26, 70, 32, 48
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=91 + act)
    OH, OW = (H - 1) // 2 + 1, (W - 1) // 2 + 1
    r = np.random.default_rng(12).standard_normal((N, OH, OW, Co)).astype(np.float32)
    buf = canary_buffer((N, OH, OW + 5, Co + 24))
    y = buf[:, :, :OW, 8:8 + Co]
    _run_s(x, w, bn, 2, act=act, residual=to_dev(r) if res_mode else None, res_mode=res_mode, y=y)
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, OW:, :]) and is_canary(buf[:, :, :OW, :8]) and is_canary(buf[:, :, :OW, 8 + Co:])


def test_halo_stride1_column_blocks(gpu, orc):
    """Images wider than one halo copy (W + 2 > 256): column blocks."""
    x, w, bn = synthetic.dense_layer(32, 48, 5, 300, N=2, k=3, seed=17)
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("case", [(16, 320, 16, 32), (16, 160, 32, 64), (16, 80, 64, 128), (32, 320, 16, 32)],
                         ids=["16-32@320-b16", "32-64@160-b16", "64-128@80-b16", "16-32@320-b32"])
def test_halo_stride2_workload_layers_sampled(gpu, orc, halo_force, case):
    """The stride-2 layers of the dense sweep and the YOLO chain at full batch on stride-2 halo
    tiles of their channel width (the cost model may send the wider ones to the im2col-path
    kernel); sampled outputs."""
    N, H, Ci, Co = case
    halo_force(str(Co))
    x, w, bn = synthetic.dense_layer(Ci, Co, H, N=N, k=3, seed=H + Ci)
    y = _run_s(x, w, bn, 2)
    idx = np.random.default_rng(Ci).choice(y.numel(), 6000, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=2, pad=1, act=orc.ACT_SILU)
    got = y.reshape(-1)[torch.from_numpy(idx).to("cuda")].cpu().numpy()
    assert rel_err(got, ref) <= TOL_TF32


@pytest.mark.parametrize("case", [(2, 9, 40, 24, 8), (1, 20, 20, 40, 32), (3, 7, 13, 24, 16), (1, 1, 1, 56, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_halo_8_channel_chunks(gpu, orc, case):
    """32-byte pixel rows with the 32-byte swizzle (Cin % 16 == 8), pixel-major 128 x 32 tiles."""
    N, H, W, Ci, Co = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case) + 5)
    y = _run(x, w, bn)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


SUB_CASES = [
    # N, H, W, Cin, Cout, stride, CB_HALO_FORCE: tiles of 2 or 4 sub-tiles of 128 pixels sharing one
    # halo copy; sub-tile counts that do not divide the tiles of a block, column blocks, 8/16/32-channel
    # chunks, stride 2
    (2, 9, 40, 32, 32, 1, "32,0,0,0,2"), (1, 20, 20, 64, 64, 1, "64,0,0,0,4"), (2, 7, 160, 16, 16, 1, "32,0,0,0,4"),
    (1, 5, 300, 16, 32, 1, "32,0,0,0,2"), (3, 11, 17, 24, 32, 1, "32,0,0,0,4"), (1, 1, 1, 32, 32, 1, "32,0,0,0,4"),
    (2, 40, 64, 16, 32, 2, "32,0,0,0,2"), (1, 21, 23, 32, 64, 2, "64,0,0,0,2"),
]


@pytest.mark.parametrize("case", SUB_CASES, ids=lambda s: "x".join(map(str, s[:6])) + "-" + s[6])
def test_halo_sub_tiles(gpu, orc, halo_force, case):
    N, H, W, Ci, Co, st, force = case
    halo_force(force)
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case[:6]) + 21)
    y = _run(x, w, bn) if st == 1 else _run_s(x, w, bn, 2)
    ref = orc.conv_bn_act(x, w, bn, stride=st, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2)])
def test_halo_sub_tiles_epilogues_and_views(gpu, orc, halo_force, act, res_mode):
    halo_force("32,0,0,0,4")
    N, H, W, Ci, Co = 2, 13, 57, 32, 24
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=71 + act)
    r = np.random.default_rng(13).standard_normal((N, H, W, Co)).astype(np.float32)
    buf = canary_buffer((N, H, W + 3, Co + 12))
    y = buf[:, :, :W, 4:4 + Co]
    _run(x, w, bn, act=act, residual=to_dev(r), res_mode=res_mode, y=y)
    ref = orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=act, residual=r, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, W:, :]) and is_canary(buf[:, :, :W, :4]) and is_canary(buf[:, :, :W, 4 + Co:])


RES_CASES = [
    # N, H, W, Cin, Cout, stride, CB_HALO_FORCE with resident weights: one channel chunk and one
    # channel tile, the nine taps copied once per CTA; sub-tiles, column blocks, stride 2, a ragged
    # channel tile, more tiles than CTAs
    (2, 20, 20, 16, 32, 1, "32,0,0,0,1,1"), (2, 21, 17, 32, 32, 1, "32,0,0,0,2,1"),
    (2, 40, 40, 16, 32, 2, "32,0,0,0,2,1"), (1, 7, 300, 16, 16, 1, "32,0,0,0,4,1"),
    (2, 12, 12, 32, 64, 1, "64,0,0,0,1,1"), (1, 9, 11, 32, 24, 1, "32,0,0,0,1,1"),
    (16, 40, 40, 32, 32, 1, "32,0,0,0,2,1"), (1, 21, 23, 16, 64, 2, "64,0,0,0,1,1"),
]


@pytest.mark.parametrize("case", RES_CASES, ids=lambda s: "x".join(map(str, s[:6])) + "-" + s[6])
def test_halo_resident_weights(gpu, orc, halo_force, case):
    N, H, W, Ci, Co, st, force = case
    halo_force(force)
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=3, seed=sum(case[:6]) + 33)
    xd = to_dev(x)
    OH, OW = (H - 1) // st + 1, (W - 1) // st + 1
    assert cb.conv_path(xd, torch.empty(N, OH, OW, Co, device="cuda"), 3, st, 1) in (cb.PATH_TC_HALO,)
    y = _run(x, w, bn) if st == 1 else _run_s(x, w, bn, 2)
    ref = orc.conv_bn_act(x, w, bn, stride=st, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


def test_halo_resident_weights_not_taken_for_several_chunks(gpu, halo_force):
    """Resident weights need one channel chunk and one channel tile: a forced request with 64 input
    channels (two 32-channel chunks) finds no plan, so the layer leaves the halo kernels."""
    halo_force("32,0,0,0,1,1")
    x = torch.empty(1, 10, 10, 64, device="cuda")
    y = torch.empty(1, 10, 10, 32, device="cuda")
    assert cb.conv_path(x, y, 3, 1, 1) not in (cb.PATH_TC_HALO, cb.PATH_TC_HALO_CM)
