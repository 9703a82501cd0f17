"""GPU parity of the depthwise-separable block run as one kernel (cb_dw_separable_block with the
one-kernel path): depthwise 3x3 + BN + ReLU kept in shared memory as the A operand of the
pointwise MMAs, the skip as identity or as a second accumulator, the final ReLU.

The pointwise and skip products are TF32 with fp32 accumulation, so the bar is the TF32 one
(5e-3 of max|oracle|) against the oracle block.  Shapes cover the four DepthwiseMNIST blocks at
two batch sizes, channel counts that leave a partial 32-channel chunk, ragged 128-pixel tiles,
256 output channels with a conv skip (two 256-column accumulators), a channel-slice output view
with padded rows, and agreement with the three-call path (kernel policy 2).
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import DwBlock
from gpu_util import TOL_TF32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def force_one_kernel():
    """Every block of these tests takes the one kernel where its shape rule allows (the default
    choice also weighs the tile count and the skip); a test may switch it off."""
    cb.set_tuning("CB_DW_BLOCK_FORCE", "1")
    yield
    cb.set_tuning("CB_DW_BLOCK_FORCE", None)


def _block_params(cin, cout, stride, seed):
    g = np.random.default_rng(seed)
    p = {"dw_w": synthetic.kaiming(g, cin, 1, 3, 3), "bn1": synthetic.bn_params(g, cin),
         "pw_w": synthetic.kaiming(g, cout, cin, 1, 1), "bn2": synthetic.bn_params(g, cout)}
    if stride != 1 or cin != cout:
        p["skip_w"] = synthetic.kaiming(g, cout, cin, 1, 1)
        p["skip_bn"] = synthetic.bn_params(g, cout)
    return p


def _run(blk, x, y, stride):
    ws = torch.empty(cb.dw_separable_block_workspace(x, y.shape[-1], stride), dtype=torch.uint8, device="cuda")
    blk(x, y, ws)
    sync_check()
    return y


CASES = [
    # N, H, Cin, Cout, stride: the MNIST blocks, then partial chunks, ragged tiles, wide outputs
    (64, 28, 48, 96, 2), (64, 14, 96, 96, 1), (64, 14, 96, 192, 2), (64, 7, 192, 192, 1),
    (3, 28, 48, 96, 2), (3, 7, 192, 192, 1),
    (2, 9, 36, 64, 2), (1, 5, 64, 64, 1), (3, 11, 100, 128, 2), (2, 7, 256, 256, 1), (1, 8, 128, 256, 2),
    (1, 1, 4, 32, 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_dw_block_one_kernel(gpu, orc, case):
    N, H, Ci, Co, s = case
    p = _block_params(Ci, Co, s, seed=sum(case))
    x = np.random.default_rng(N * H + Ci).standard_normal((N, H, H, Ci)).astype(np.float32)
    blk = DwBlock(p, Ci, Co, s)
    OH = (H - 1) // s + 1
    y = torch.empty(N, OH, OH, Co, device="cuda")
    xd = to_dev(x)
    assert cb.dw_separable_block_fused(xd, blk.params, y)
    _run(blk, xd, y, s)
    ref = orc.dw_separable_block(x, p, s)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32


@pytest.mark.parametrize("case", [(64, 28, 48, 96, 2), (64, 7, 192, 192, 1), (3, 11, 100, 128, 2)],
                         ids=lambda c: "x".join(map(str, c)))
def test_dw_block_one_kernel_matches_three_calls(gpu, case):
    """The one kernel against the depthwise, skip and pointwise layers run one by one (policy 2):
    the same TF32 products, rounded at different points (the three-call path stores the depthwise
    and skip outputs in memory), so they agree to the TF32 bar."""
    N, H, Ci, Co, s = case
    p = _block_params(Ci, Co, s, seed=3 + Ci)
    x = to_dev(np.random.default_rng(5).standard_normal((N, H, H, Ci)).astype(np.float32))
    blk = DwBlock(p, Ci, Co, s)
    OH = (H - 1) // s + 1
    y0 = _run(blk, x, torch.empty(N, OH, OH, Co, device="cuda"), s)
    cb.set_kernel_policy(2)
    try:
        y1 = torch.empty_like(y0)
        assert not cb.dw_separable_block_fused(x, blk.params, y1)
        _run(blk, x, y1, s)
    finally:
        cb.set_kernel_policy(0)
    assert rel_err(y0.cpu().numpy(), y1.cpu().numpy()) <= TOL_TF32


def test_dw_block_one_kernel_output_view(gpu, orc):
    """Output into channels [32, 32 + Co) of a wider buffer with padded rows: nothing else written."""
    N, H, Ci, Co, s = 2, 10, 64, 96, 2
    p = _block_params(Ci, Co, s, seed=9)
    x = np.random.default_rng(9).standard_normal((N, H, H, Ci)).astype(np.float32)
    blk = DwBlock(p, Ci, Co, s)
    OH = (H - 1) // s + 1
    buf = canary_buffer((N, OH, OH + 3, Co + 64))
    y = buf[:, :, :OH, 32:32 + Co]
    xd = to_dev(x)
    assert cb.dw_separable_block_fused(xd, blk.params, y)
    _run(blk, xd, y, s)
    assert rel_err(y.cpu().numpy(), orc.dw_separable_block(x, p, s)) <= TOL_TF32
    assert is_canary(buf[:, :, OH:, :]) and is_canary(buf[:, :, :OH, :32]) and is_canary(buf[:, :, :OH, 32 + Co:])


def test_dw_block_one_kernel_not_taken(gpu):
    p = _block_params(48, 40, 2, seed=1)  # Co % 32 != 0
    blk = DwBlock(p, 48, 40, 2)
    x = torch.empty(1, 8, 8, 48, device="cuda")
    assert not cb.dw_separable_block_fused(x, blk.params, torch.empty(1, 4, 4, 40, device="cuda"))
    p = _block_params(48, 96, 2, seed=1)
    blk = DwBlock(p, 48, 96, 2)
    xs = torch.empty(1, 8, 8, 50, device="cuda")[..., 1:49]  # pixels not 16-byte aligned
    assert not cb.dw_separable_block_fused(xs, blk.params, torch.empty(1, 4, 4, 96, device="cuda"))


def test_dw_block_default_choice(gpu):
    """Without the override: one kernel for a conv-skip block with at least 64 tiles, three layer
    kernels for identity blocks and small grids."""
    cb.set_tuning("CB_DW_BLOCK_FORCE", None)
    p = _block_params(48, 96, 2, seed=1)
    blk = DwBlock(p, 48, 96, 2)
    x = torch.empty(64, 28, 28, 48, device="cuda")  # 64 x 14 x 14 outputs: 98 tiles
    assert cb.dw_separable_block_fused(x, blk.params, torch.empty(64, 14, 14, 96, device="cuda"))
    x = torch.empty(8, 28, 28, 48, device="cuda")  # 13 tiles
    assert not cb.dw_separable_block_fused(x, blk.params, torch.empty(8, 14, 14, 96, device="cuda"))
    p = _block_params(96, 96, 1, seed=2)
    blk = DwBlock(p, 96, 96, 1)
    x = torch.empty(64, 14, 14, 96, device="cuda")  # identity skip
    assert not cb.dw_separable_block_fused(x, blk.params, torch.empty(64, 14, 14, 96, device="cuda"))
