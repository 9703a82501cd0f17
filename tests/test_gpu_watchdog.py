"""The failure path of the bounded waits, on the GPU, without a hang or a fault.

cb_debug_timeout_probe launches a CTA whose mbarrier wait nothing satisfies; the wait gives up
after the given limit through the same watchdog every pipeline kernel uses.  The device error
word must then read CB_ERR_TIMEOUT once (and be cleared by reading it), and the context must stay
usable: a layer launched afterwards still matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, TOL_TF32, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(gpu, orc):
    assert cb.get_device_error() == cb.OK
    t0 = time.perf_counter()
    cb.debug_timeout_probe(20)
    assert cb.get_device_error() == cb.ERR_TIMEOUT
    assert time.perf_counter() - t0 < 5.0
    assert cb.get_device_error() == cb.OK  # reading cleared it
    x, w, bn = synthetic.dense_layer(8, 16, 12, N=1, k=3, seed=3)
    y = torch.empty(1, 12, 12, 16, device="cuda")
    ConvBnAct(w, bn, 1, 1, cb.ACT_RELU)(to_dev(x), y)
    sync_check()
    tol = TOL_TF32 if cb.layer_uses_tensor_cores(8, 16, 3, 1) else TOL_FP32
    assert rel_err(y.cpu().numpy(), orc.conv_bn_act(x, w, bn, stride=1, pad=1, act=orc.ACT_RELU)) <= tol


def test_timeout_probe_rejects_bad_limits(gpu):
    for bad in (0, -1, 10001):
        with pytest.raises(cb.CbError):
            cb.debug_timeout_probe(bad)


@pytest.mark.parametrize("stride", [1, 2])
def test_depthwise_pipeline_wait_runs_out(gpu, orc, stride):
    """Inside a real pipeline: the TMA depthwise kernel's producer withholds one row (fault
    injection through CB_DEBUG_DW_SKIP_ROW, nothing is issued against that barrier), so the
    consumers' bounded wait runs out after CB_TIMEOUT_MS.  The kernel records CB_ERR_TIMEOUT,
    drains its copies, frees nothing it does not hold and returns: no hang, no fault.  The error
    reads once, and the same layer run again without the injection matches the oracle."""
    x, w, bn = synthetic.depthwise_layer(2, 64, 20, 20, seed=stride)
    layer = ConvBnAct(w, bn, stride, 1, cb.ACT_RELU, groups=64)
    OH, OW = layer.out_hw(20, 20)
    xd = to_dev(x)
    y = torch.empty(2, OH, OW, 64, device="cuda")
    assert cb.get_device_error() == cb.OK
    with cb.tuning("CB_TIMEOUT_MS", "50"), cb.tuning("CB_DEBUG_DW_SKIP_ROW", "1"):
        t0 = time.perf_counter()
        layer(xd, y)
        assert "dw_tma_kernel" in cb.last_launch()["kernel"]
        assert cb.get_device_error() == cb.ERR_TIMEOUT
        assert time.perf_counter() - t0 < 5.0
    assert cb.get_device_error() == cb.OK  # reading cleared it
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=stride, pad=1, groups=64, act=orc.ACT_RELU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_stage_body_tc_wait_runs_out(gpu, orc):
    """Inside the tensor-core stage body (32 channels): no warpgroup issues the copy or the barrier
    arrive of its first x1 tile (fault injection through CB_DEBUG_STAGE_SKIP_X, nothing is issued
    against that barrier), so each first wait runs out after CB_TIMEOUT_MS or sees the CTA's abort
    flag.  The kernel records CB_ERR_TIMEOUT, frees its tensor memory and returns: no hang, no
    fault.  The error reads once, and the same body run again without the injection matches the
    oracle."""
    from conv_bn_activation_gb300.nets import ConvBnAct as L
    from gpu_util import oracle_stage_body
    st = synthetic.yolo_params()[1]
    layers = [L(st[k + "_w"], st[k + "_bn"], 1, p, cb.ACT_SILU) for k, p in (("cv1", 0), ("cv2", 1), ("cv3", 0))]
    x1 = np.random.default_rng(11).standard_normal((2, 20, 40, 32)).astype(np.float32)
    xd = to_dev(x1)
    y = torch.empty(2, 20, 40, 32, device="cuda")
    assert cb.get_device_error() == cb.OK
    with cb.tuning("CB_TIMEOUT_MS", "50"), cb.tuning("CB_DEBUG_STAGE_SKIP_X", "1"):
        t0 = time.perf_counter()
        cb.stage_body(xd, layers, cb.ACT_SILU, y)
        assert "stage_body_tc_kernel" in cb.last_launch()["kernel"]
        assert cb.get_device_error() == cb.ERR_TIMEOUT
        assert time.perf_counter() - t0 < 5.0
    assert cb.get_device_error() == cb.OK  # reading cleared it
    cb.stage_body(xd, layers, cb.ACT_SILU, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_TF32
