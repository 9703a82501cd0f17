"""Shared helpers for the GPU parity tests (no arithmetic of the method here)."""
import numpy as np
import torch

from conv_bn_activation_gb300 import binding as cb

TOL_FP32 = 1e-5   # CUDA-core fp32 kernels: max|gpu - oracle| / max|oracle|
TOL_TF32 = 5e-3   # tensor-core TF32 kernels with fp32 accumulate


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (scale if scale > 0 else 1.0))


def to_dev(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def canary_buffer(shape, device="cuda"):
    """A float32 buffer filled with a NaN bit pattern no kernel produces."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.view(torch.int32).fill_(0x7FC0DEAD)
    return t


def is_canary(t):
    return bool((t.contiguous().view(torch.int32) == 0x7FC0DEAD).all().item())


def sync_check():
    torch.cuda.synchronize()
    assert cb.get_device_error() == cb.OK
