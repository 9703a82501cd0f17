"""The allocation-free depthwise-separable block (cb_dw_separable_block_static).

It exists for callers that cannot allocate device memory where they run a
block (a host framework that owns all device memory, a real-time loop that
must not allocate after start-up, a plain C host without an allocator).  Its
scratch is a fixed file-scope device array instead of a caller workspace.
Its output must equal the workspace entry point's, call after call, even
though the array keeps the previous call's contents.  This file is collected
last so that a failure here cannot hide failures elsewhere.
"""
import ctypes

import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import DwBlock
from gpu_util import TOL_TF32, rel_err, sync_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("blk_index", [0, 1, 2, 3])
def test_static_block_matches_workspace_block_twice(gpu, blk_index):
    params = synthetic.mnist_params()
    cin, cout, s = synthetic.MNIST_BLOCKS[blk_index]
    H = (28, 14, 14, 7)[blk_index]
    OH = (H - 1) // s + 1
    blk = DwBlock(params["blocks"][blk_index], cin, cout, s)
    g = np.random.default_rng(blk_index)
    for call in range(2):
        # a fresh input each time: the array still holds the previous call's t and s
        x = torch.from_numpy(g.standard_normal((64, H, H, cin)).astype(np.float32)).to(gpu)
        ws = torch.empty(cb.dw_separable_block_workspace(x, cout, s), dtype=torch.uint8, device=gpu)
        y_ref = torch.empty(64, OH, OH, cout, device=gpu)
        blk(x, y_ref, ws)
        y = torch.full((64, OH, OH, cout), float("nan"), device=gpu)
        st = cb.dw_separable_block_static(x, blk.params, s, y)
        assert st == cb.OK, cb.status_string(st)
        sync_check()
        assert rel_err(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL_TF32, f"call {call}"


def test_static_block_rejects_oversize(gpu):
    """A block whose scratch would exceed the fixed array is refused before anything runs."""
    params = synthetic.mnist_params()
    blk = DwBlock(params["blocks"][0], 48, 96, 2)
    N = 1024  # t alone is 1024*14*14*48*4 bytes = 38.5 MB > 16 MiB
    x = torch.empty(N, 28, 28, 48, device=gpu)
    y = torch.empty(N, 14, 14, 96, device=gpu)
    assert cb.dw_separable_block_workspace(x, 96, 2) > cb.STATIC_SCRATCH_BYTES
    assert cb.dw_separable_block_static(x, blk.params, 2, y) == cb.ERR_WORKSPACE
