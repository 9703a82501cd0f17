"""The allocation-free depthwise-separable block (cb_dw_separable_block_static).

Some callers cannot call cudaMalloc where they run a block: a host framework
that owns all device memory, a real-time loop that must not allocate after
start-up, a plain C host linked without an allocator.  For them the block's
scratch (the depthwise output t and the skip output s) lives in a fixed
file-scope device array instead of a caller workspace.

These tests force the three-layer path of the block (CB_DW_BLOCK_FORCE=0),
which is the one that goes through the scratch, so every case writes and
reads the array.  On two calls in a row with fresh inputs (the array still
holds the previous call's t and s) the output must equal the workspace entry
point's bit for bit (the same kernels on another buffer) and match the
oracle's DepthwiseSeparableConv within the tensor-core bar.  This file is
collected last so that a failure here cannot hide failures elsewhere; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import DwBlock
from gpu_util import TOL_TF32, rel_err, sync_check

pytestmark = pytest.mark.gpu


@pytest.fixture
def layered_path():
    """The block as three layer kernels through the scratch (the one-kernel path uses none)."""
    with cb.tuning("CB_DW_BLOCK_FORCE", "0"):
        yield


@pytest.mark.parametrize("blk_index", [0, 1, 2, 3])
def test_static_block_matches_workspace_and_oracle_twice(gpu, orc, layered_path, blk_index):
    params = synthetic.mnist_params()
    p = params["blocks"][blk_index]
    cin, cout, s = synthetic.MNIST_BLOCKS[blk_index]
    H = (28, 14, 14, 7)[blk_index]
    OH = (H - 1) // s + 1
    blk = DwBlock(p, cin, cout, s)
    g = np.random.default_rng(blk_index)
    for call in range(2):
        # a fresh input each time: the array still holds the previous call's t and s
        x_host = g.standard_normal((64, H, H, cin)).astype(np.float32)
        x = torch.from_numpy(x_host).to(gpu)
        y_ws = torch.empty(64, OH, OH, cout, device=gpu)
        assert not cb.dw_separable_block_fused(x, blk.params, y_ws)
        ws = torch.empty(cb.dw_separable_block_workspace(x, cout, s), dtype=torch.uint8, device=gpu)
        blk(x, y_ws, ws)
        y = torch.full((64, OH, OH, cout), float("nan"), device=gpu)
        st = cb.dw_separable_block_static(x, blk.params, s, y)
        assert st == cb.OK, cb.status_string(st)
        sync_check()
        got = y.cpu().numpy()
        assert np.array_equal(got, y_ws.cpu().numpy()), f"call {call}: differs from the workspace path"
        ref = orc.dw_separable_block(x_host, p, s)
        assert rel_err(got, ref) <= TOL_TF32, f"call {call}"


def test_static_block_rejects_oversize(gpu):
    """A block whose scratch would exceed the fixed array is refused before anything runs."""
    params = synthetic.mnist_params()
    blk = DwBlock(params["blocks"][0], 48, 96, 2)
    N = 1024  # t alone is 1024*14*14*48*4 bytes = 38.5 MB > 16 MiB
    x = torch.empty(N, 28, 28, 48, device=gpu)
    y = torch.empty(N, 14, 14, 96, device=gpu)
    assert cb.dw_separable_block_workspace(x, 96, 2) > cb.STATIC_SCRATCH_BYTES
    assert cb.dw_separable_block_static(x, blk.params, 2, y) == cb.ERR_WORKSPACE
