"""GPU parity of the im2col-path tensor-core kernel with pixel-block tiles: tiles of blk_h x blk_w
output pixels of one image whose A operand is one tiled copy per (filter tap, channel chunk),
traversed with element strides equal to the conv stride (CB_IGEMM_BLOCKS=1 forces them where the
shape allows; by default they are used when they waste at most 15 % of the tile rows).

Shapes: 3x3 and 1x1, stride 1 and 2, 8-, 16- and 32-channel chunks, blocks that fit the output
exactly and ragged ones, images smaller than a block, residuals, channel-slice output views with
padded rows; each against the fp64 oracle at the TF32 bar, and against the im2col-mode tiles.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_TF32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def no_halo_tiles():
    """Policy 2 (tensor cores without the halo kernel) keeps every case on the im2col-path kernel."""
    cb.set_kernel_policy(2)
    yield
    cb.set_kernel_policy(0)


@pytest.fixture
def blocks_mode():
    cb.set_tuning("CB_IGEMM_BLOCKS", None)
    yield lambda v: cb.set_tuning("CB_IGEMM_BLOCKS", v)
    cb.set_tuning("CB_IGEMM_BLOCKS", None)


CASES = [
    # N, H, W, Cin, Cout, k, stride
    (2, 32, 64, 32, 64, 3, 2), (1, 40, 40, 16, 32, 3, 2), (2, 20, 24, 40, 48, 3, 1), (1, 16, 16, 8, 48, 1, 1),
    (2, 10, 50, 64, 96, 1, 1), (1, 21, 37, 32, 40, 1, 2), (1, 7, 7, 32, 32, 3, 2), (3, 9, 130, 24, 16, 3, 1),
]


def _layer_out(case, seed, act=cb.ACT_SILU, residual=None, res_mode=0, y=None, paths=(cb.PATH_TC_IM2COL,)):
    N, H, W, Ci, Co, k, s = case
    x, w, bn = synthetic.dense_layer(Ci, Co, H, W, N=N, k=k, seed=seed)
    layer = ConvBnAct(w, bn, s, k // 2, act)
    OH, OW = layer.out_hw(H, W)
    if y is None:
        y = torch.empty(N, OH, OW, Co, device="cuda")
    xd = to_dev(x)
    assert cb.conv_path(xd, y, k, s, k // 2) in paths
    layer(xd, y, residual=residual, res_mode=res_mode)
    sync_check()
    return x, w, bn, y


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_pixel_blocks(gpu, orc, blocks_mode, case):
    blocks_mode("1")
    N, H, W, Ci, Co, k, s = case
    x, w, bn, y = _layer_out(case, seed=sum(case))
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=k // 2, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    # the same products in im2col-mode tiles: rounded outputs may differ in the last stored bit
    blocks_mode("0")
    _, _, _, y0 = _layer_out(case, seed=sum(case))
    assert rel_err(y.cpu().numpy(), y0.cpu().numpy()) <= 2.0 ** -10


@pytest.mark.parametrize("act,res_mode", [(1, 1), (2, 2), (0, 0)])
def test_pixel_blocks_epilogues_and_views(gpu, orc, blocks_mode, act, res_mode):
    """Blocks that overhang the output on both edges, into a channel slice of a padded buffer."""
    blocks_mode("1")
    case = (2, 26, 70, 32, 48, 3, 2)
    N, H, W, Ci, Co, k, s = case
    OH, OW = (H - 1) // 2 + 1, (W - 1) // 2 + 1
    r = np.random.default_rng(3).standard_normal((N, OH, OW, Co)).astype(np.float32)
    buf = canary_buffer((N, OH, OW + 5, Co + 24))
    yv = buf[:, :, :OW, 8:8 + Co]
    x, w, bn, y = _layer_out(case, seed=77 + act, act=act, residual=to_dev(r) if res_mode else None,
                             res_mode=res_mode, y=yv)
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert is_canary(buf[:, :, OW:, :]) and is_canary(buf[:, :, :OW, :8]) and is_canary(buf[:, :, :OW, 8 + Co:])


@pytest.mark.parametrize("case", [(16, 320, 320, 16, 32, 3, 2), (32, 160, 160, 16, 16, 3, 1)],
                         ids=["dense-16-32@320s2-b16", "yolo-16-16@160-b32"])
def test_pixel_blocks_workload_layers_sampled(gpu, orc, case):
    """The 16-channel layers of the dense sweep and the YOLO chain at full batch on the im2col-path
    kernel (the benchmarks run them on halo tiles); sampled outputs."""
    N, H, W, Ci, Co, k, s = case
    x, w, bn, y = _layer_out(case, seed=5)
    idx = np.random.default_rng(Ci + H).choice(y.numel(), 6000, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=s, pad=1, act=orc.ACT_SILU)
    got = y.reshape(-1)[torch.from_numpy(idx).to("cuda")].cpu().numpy()
    assert rel_err(got, ref) <= TOL_TF32
