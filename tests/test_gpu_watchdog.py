"""The failure path of the bounded waits, on the GPU, without a hang or a fault.

cb_debug_timeout_probe launches a CTA whose mbarrier wait nothing satisfies; the wait gives up
after the given limit through the same watchdog every pipeline kernel uses.  The device error
word must then read CB_ERR_TIMEOUT once (and be cleared by reading it), and the context must stay
usable: a layer launched afterwards still matches the oracle.
"""
import time

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
