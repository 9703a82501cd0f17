"""Shared helpers for the GPU parity tests (no arithmetic of the method here)."""
import numpy as np
import torch

from conv_bn_activation_gb300 import binding as cb

TOL_FP32 = 1e-5   # CUDA-core fp32 kernels: max|gpu - oracle| / max|oracle|
TOL_TF32 = 5e-3   # tensor-core TF32 kernels with fp32 accumulate
TOL_BF16 = 5e-3   # bf16 storage (fp32 arithmetic): max|gpu - oracle| / max|oracle|


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


def to_dev_bf16(a, device="cuda"):
    """(bf16 device tensor, the fp32 numpy array of its exact values): the input the kernel and
    the oracle both see."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.to(device), t.float().numpy()


def bf16_within_half_ulp(got, ref):
    """max over elements of |got - ref| / (2^-8 |ref| + 1e-5 max|ref|): at most 1 when every
    output is the fp32 result rounded to bf16 (half a unit in the last of bf16's 8 significant
    bits is at most 2^-8 of the value) up to fp32 arithmetic error."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got))
    bound = 2.0 ** -8 * np.abs(ref) + TOL_FP32 * max(float(np.max(np.abs(ref))), 1e-30)
    return float(np.max(np.abs(got - ref) / bound))


def canary_buffer_bf16(shape, device="cuda"):
    """A bf16 buffer filled with a NaN bit pattern no kernel produces."""
    t = torch.empty(shape, dtype=torch.bfloat16, device=device)
    t.view(torch.int16).fill_(0x7FDD)
    return t


def is_canary_bf16(t):
    return bool((t.contiguous().view(torch.int16) == 0x7FDD).all().item())


def stage_body_tol(c):
    """The bar of cb_stage_body at C channels: fp32 on the CUDA cores (16), TF32 on the tensor cores (32)."""
    return TOL_FP32 if c == 16 else TOL_TF32


def to_bf16_values(a):
    """The bf16 values (nearest even) of an array, as float32."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def oracle_stage_body_bf16_storage(orc, x1, st, act=2):
    """The stage body as its three layers compute it with bf16 storage: the oracle's layers composed,
    with a and b rounded to bf16 where the layers store them and the 3x3's weights rounded to bf16
    as the bf16 tensor-core layer multiplies them (the 1x1 layers multiply fp32 weights)."""
    a = to_bf16_values(orc.conv_bn_act(x1, st["cv1_w"], st["cv1_bn"], stride=1, pad=0, act=act))
    b = to_bf16_values(orc.conv_bn_act(a, to_bf16_values(st["cv2_w"]), st["cv2_bn"], stride=1, pad=1, act=act))
    cat = np.ascontiguousarray(np.concatenate([a, b], axis=-1))
    return orc.conv_bn_act(cat, st["cv3_w"], st["cv3_bn"], stride=1, pad=0, act=act, residual=x1,
                           res_mode=orc.RES_POST_ACT)


def oracle_stage_body(orc, x1, st, act=2):
    """The oracle's YOLO-style stage body from its stride-2 output x1 (NHWC): cv1 (1x1), cv2 (3x3,
    pad 1) on cv1's output, cv3 (1x1) on the concat [a | b] with x1 added after the activation --
    the three layers' definitions composed (the stage of oracle.yolo_stage after its down conv)."""
    a = orc.conv_bn_act(x1, st["cv1_w"], st["cv1_bn"], stride=1, pad=0, act=act)
    b = orc.conv_bn_act(a, st["cv2_w"], st["cv2_bn"], stride=1, pad=1, act=act)
    cat = np.ascontiguousarray(np.concatenate([a, b], axis=-1))
    return orc.conv_bn_act(cat, st["cv3_w"], st["cv3_bn"], stride=1, pad=0, act=act, residual=x1,
                           res_mode=orc.RES_POST_ACT)
