"""Thin Python binding over the C ABI in include/cb.h (ctypes).

Argument marshalling only: every step of the computation runs in libcb.so's
CUDA kernels.  torch supplies device memory and streams.  If libcb.so is
missing or cannot be loaded, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcb.so")
_lib = None
_lock = threading.Lock()

# enums (include/cb.h)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIGNMENT, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = range(7)
ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2
RES_NONE, RES_PRE_ACT, RES_POST_ACT = 0, 1, 2
LAYOUT_NHWC, LAYOUT_NCHW = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1
PATH_DIRECT, PATH_DEPTHWISE, PATH_TC_IM2COL, PATH_TC_HALO, PATH_TC_HALO_CM, PATH_POINTWISE, PATH_STEM = range(1, 8)

EXPORTED = (
    "cb_fold_bn", "cb_repack_weights", "cb_conv_bn_act", "cb_dw_separable_block_workspace",
    "cb_dw_separable_block", "cb_avgpool_linear", "cb_preprocess_u8", "cb_preprocess_u8_three_pass",
    "cb_get_device_error", "cb_last_cuda_error", "cb_set_kernel_policy", "cb_status_string", "cb_version",
    "cb_round_weights_tf32", "cb_get_kernel_policy", "cb_layer_uses_tensor_cores",
    "cb_dw_separable_block_static", "cb_conv_path", "cb_debug_timeout_probe", "cb_autotune_conv",
    "cb_autotune_clear", "cb_autotune_entries", "cb_preprocess_stem_u8", "cb_dw_separable_block_fused",
    "cb_set_tuning", "cb_last_launch", "cb_debug_sample_coords", "cb_convert_weights_bf16", "cb_stage_body",
)
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024  # CB_STATIC_SCRATCH_BYTES


class CbTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("n", ctypes.c_int), ("h", ctypes.c_int), ("w", ctypes.c_int), ("c", ctypes.c_int),
        ("stride_n", ctypes.c_longlong), ("stride_h", ctypes.c_longlong),
        ("stride_w", ctypes.c_longlong), ("stride_c", ctypes.c_longlong),
        ("layout", ctypes.c_int), ("dtype", ctypes.c_int),
    ]


class CbLaunchInfo(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int), ("threads", ctypes.c_int), ("smem_bytes", ctypes.c_size_t),
                ("cluster", ctypes.c_int), ("blocks_per_sm", ctypes.c_int), ("kernel", ctypes.c_char_p)]


class CbError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {status_string(status)}"
        if status == ERR_CUDA:
            msg += f" (cudaError {load().cb_last_cuda_error()})"
        super().__init__(msg)


def load():
    """Load libcb.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"libcb.so not built ({_LIB_PATH}); run __graft_entry__.build()")
            lib = ctypes.CDLL(_LIB_PATH)
            P, I, F, LL, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong, ctypes.c_size_t
            T = ctypes.POINTER(CbTensor)
            sig = {
                "cb_fold_bn": [P, P, P, P, F, I, P, P],
                "cb_repack_weights": [P, I, I, I, I, I, P],
                "cb_conv_bn_act": [T, P, P, P, I, I, I, I, I, I, T, I, T, P],
                "cb_dw_separable_block_workspace": [T, I, I, ctypes.POINTER(S)],
                "cb_dw_separable_block": [T, P, P, P, P, P, P, P, P, P, I, T, P, S, P],
                "cb_dw_separable_block_static": [T, P, P, P, P, P, P, P, P, P, I, T, P],
                "cb_stage_body": [T, P, P, P, P, P, P, P, P, P, I, T, P],
                "cb_avgpool_linear": [T, P, P, I, P, P],
                "cb_preprocess_u8": [P, I, I, I, LL, P, I, I, P],
                "cb_preprocess_u8_three_pass": [P, I, I, I, LL, P, P, P, I, I, P],
                "cb_get_device_error": [P],
                "cb_last_cuda_error": [],
                "cb_set_kernel_policy": [I],
                "cb_get_kernel_policy": [],
                "cb_round_weights_tf32": [P, LL, P],
                "cb_convert_weights_bf16": [P, LL, P],
                "cb_layer_uses_tensor_cores": [I, I, I, I, I],
                "cb_conv_path": [T, T, I, I, I, I],
                "cb_debug_timeout_probe": [I, P],
                "cb_debug_sample_coords": [I, I, P, P, P, P],
                "cb_autotune_conv": [T, P, P, P, I, I, I, I, I, I, T, I, T, P],
                "cb_autotune_clear": [],
                "cb_preprocess_stem_u8": [P, I, I, I, LL, I, I, P, P, P, I, T, P],
                "cb_dw_separable_block_fused": [T, T, P, P],
                "cb_autotune_entries": [],
                "cb_set_tuning": [ctypes.c_char_p, ctypes.c_char_p],
                "cb_last_launch": [ctypes.POINTER(CbLaunchInfo)],
                "cb_status_string": [I],
                "cb_version": [],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_char_p if name == "cb_status_string" else ctypes.c_int
            _lib = lib
    return _lib


def status_string(s: int) -> str:
    return load().cb_status_string(int(s)).decode()


def _check(status: int, where: str):
    if status != OK:
        raise CbError(status, where)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ----------------------------------------------------------------- views
def dtype_code(t) -> int:
    """cb_dtype of a torch tensor: float32 -> DTYPE_F32, bfloat16 -> DTYPE_BF16."""
    import torch
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"activation tensors are float32 or bfloat16, got {t.dtype}")


def nhwc(t, n=None, h=None, w=None, c=None) -> CbTensor:
    """View of a torch tensor indexed [N, H, W, C] (any strides, unit channel stride)."""
    N, H, W, C = t.shape
    sn, sh, sw, sc = t.stride()
    return CbTensor(t.data_ptr(), N if n is None else n, H if h is None else h, W if w is None else w,
                    C if c is None else c, sn, sh, sw, sc, LAYOUT_NHWC, dtype_code(t))


def nchw(t) -> CbTensor:
    """View of a torch tensor indexed [N, C, H, W] (unit W stride)."""
    N, C, H, W = t.shape
    sn, sc, sh, sw = t.stride()
    return CbTensor(t.data_ptr(), N, H, W, C, sn, sh, sw, sc, LAYOUT_NCHW, dtype_code(t))


# ----------------------------------------------------------- host helpers
def fold_bn(gamma, beta, mean, var, eps=1e-5):
    """cb_fold_bn on host arrays -> (scale, bias) float32 numpy arrays."""
    g, b, m, v = (np.ascontiguousarray(a, dtype=np.float32) for a in (gamma, beta, mean, var))
    C = g.size
    scale = np.empty(C, np.float32)
    bias = np.empty(C, np.float32)
    _check(load().cb_fold_bn(g.ctypes.data, b.ctypes.data, m.ctypes.data, v.ctypes.data, ctypes.c_float(eps), C,
                             scale.ctypes.data, bias.ctypes.data), "cb_fold_bn")
    return scale, bias


def repack_weights(w_oihw, groups=1):
    """cb_repack_weights: OIHW -> OHWI (dense) or [kh, kw, C] (depthwise), host numpy."""
    w = np.ascontiguousarray(w_oihw, dtype=np.float32)
    Co, cig, kh, kw = w.shape
    out = np.empty(w.size, np.float32)
    _check(load().cb_repack_weights(w.ctypes.data, Co, cig, kh, kw, groups, out.ctypes.data), "cb_repack_weights")
    if groups == 1:
        return out.reshape(Co, kh, kw, cig)
    return out.reshape(kh, kw, Co)


def set_kernel_policy(policy: int):
    _check(load().cb_set_kernel_policy(policy), "cb_set_kernel_policy")


def get_kernel_policy() -> int:
    return load().cb_get_kernel_policy()


def set_tuning(name: str, value=None):
    """cb_set_tuning: set a plan override (CB_HALO_FORCE, CB_IGEMM_FORCE, ...); None restores the default."""
    _check(load().cb_set_tuning(name.encode(), None if value is None else str(value).encode()), "cb_set_tuning")


class tuning:
    """Context manager: a plan override for the calls inside the block, restored to the default on exit."""

    def __init__(self, name: str, value):
        self.name, self.value = name, value

    def __enter__(self):
        set_tuning(self.name, self.value)
        return self

    def __exit__(self, *exc):
        set_tuning(self.name, None)
        return False


def last_launch() -> dict:
    """cb_last_launch: launch configuration, occupancy (CTAs per SM) and name of this thread's last kernel."""
    info = CbLaunchInfo()
    _check(load().cb_last_launch(ctypes.byref(info)), "cb_last_launch")
    return {"grid": info.grid, "threads": info.threads, "smem_bytes": int(info.smem_bytes), "cluster": info.cluster,
            "blocks_per_sm": info.blocks_per_sm, "kernel": (info.kernel or b"?").decode()}


def round_weights_tf32(w):
    """cb_round_weights_tf32 on a host array (any shape) -> rounded float32 copy."""
    a = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty_like(a)
    _check(load().cb_round_weights_tf32(a.ctypes.data, a.size, out.ctypes.data), "cb_round_weights_tf32")
    return out


def convert_weights_bf16(w):
    """cb_convert_weights_bf16 on a host array (any shape) -> torch.bfloat16 CPU tensor of the same shape."""
    import torch
    a = np.ascontiguousarray(w, dtype=np.float32)
    out = np.empty(a.shape, np.uint16)
    _check(load().cb_convert_weights_bf16(a.ctypes.data, a.size, out.ctypes.data), "cb_convert_weights_bf16")
    return torch.from_numpy(out.view(np.int16)).view(torch.bfloat16)


def layer_uses_tensor_cores(ci, co, k, stride=1, groups=1) -> bool:
    """cb_layer_uses_tensor_cores: the layer computes in TF32 on the tensor cores (round its weights)."""
    return bool(load().cb_layer_uses_tensor_cores(ci, co, k, stride, groups))


def conv_path(x, y, k, stride, pad, groups=1, x_layout=LAYOUT_NHWC) -> int:
    """cb_conv_path: which kernel cb_conv_bn_act would run (PATH_*), 0 if unsupported."""
    xv = nchw(x) if x_layout == LAYOUT_NCHW else nhwc(x)
    yv = nhwc(y)
    return load().cb_conv_path(ctypes.byref(xv), ctypes.byref(yv), k, stride, pad, groups)


def version() -> int:
    return load().cb_version()


# ------------------------------------------------------------- GPU calls
def conv_bn_act(x, w, scale, bias, k, stride, pad, groups, act, y, residual=None, res_mode=RES_NONE,
                stream=None, x_layout=LAYOUT_NHWC):
    """cb_conv_bn_act on torch CUDA tensors.  x: [N,H,W,C] (or [N,C,H,W] with
    x_layout=LAYOUT_NCHW); y, residual: [N,OH,OW,Co] views; w, scale, bias:
    device tensors in the cb_repack_weights / cb_fold_bn layouts.  x, y and
    residual are float32, or all bfloat16 for the layers that take bf16
    storage (depthwise 3x3, narrow 1x1); weights, scale and bias stay float32."""
    xv = nchw(x) if x_layout == LAYOUT_NCHW else nhwc(x)
    yv = nhwc(y)
    rv = nhwc(residual) if residual is not None else None
    st = load().cb_conv_bn_act(ctypes.byref(xv), w.data_ptr(), scale.data_ptr(), bias.data_ptr(), k, k, stride, pad,
                               groups, act, ctypes.byref(rv) if rv is not None else None, res_mode,
                               ctypes.byref(yv), _stream_ptr(stream))
    _check(st, "cb_conv_bn_act")
    return y


def autotune_conv(x, w, scale, bias, k, stride, pad, groups, act, y, residual=None, res_mode=RES_NONE,
                  stream=None, x_layout=LAYOUT_NHWC):
    """cb_autotune_conv: time the layer's tile plans on these buffers, keep the fastest for the
    shape; y holds the result.  Synchronises the stream (not inside graph capture)."""
    xv = nchw(x) if x_layout == LAYOUT_NCHW else nhwc(x)
    yv = nhwc(y)
    rv = nhwc(residual) if residual is not None else None
    st = load().cb_autotune_conv(ctypes.byref(xv), w.data_ptr(), scale.data_ptr(), bias.data_ptr(), k, k, stride,
                                 pad, groups, act, ctypes.byref(rv) if rv is not None else None, res_mode,
                                 ctypes.byref(yv), _stream_ptr(stream))
    _check(st, "cb_autotune_conv")
    return y


def autotune_clear():
    load().cb_autotune_clear()


def autotune_entries() -> int:
    return load().cb_autotune_entries()


def dw_separable_block_workspace(x, c_out, stride) -> int:
    xv = nhwc(x)
    n = ctypes.c_size_t(0)
    _check(load().cb_dw_separable_block_workspace(ctypes.byref(xv), c_out, stride, ctypes.byref(n)),
           "cb_dw_separable_block_workspace")
    return n.value


def dw_separable_block(x, p, stride, y, workspace, stream=None):
    """p: dict of device tensors dw_w, dw_scale, dw_bias, pw_w, pw_scale, pw_bias and optionally
    skip_w, skip_scale, skip_bias.  workspace: uint8 device tensor."""
    xv, yv = nhwc(x), nhwc(y)
    sk = p.get("skip_w")
    st = load().cb_dw_separable_block(
        ctypes.byref(xv), p["dw_w"].data_ptr(), p["dw_scale"].data_ptr(), p["dw_bias"].data_ptr(),
        p["pw_w"].data_ptr(), p["pw_scale"].data_ptr(), p["pw_bias"].data_ptr(),
        sk.data_ptr() if sk is not None else None,
        p["skip_scale"].data_ptr() if sk is not None else None,
        p["skip_bias"].data_ptr() if sk is not None else None,
        stride, ctypes.byref(yv), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
        _stream_ptr(stream))
    _check(st, "cb_dw_separable_block")
    return y


def stage_body(x1, layers, act, y, stream=None):
    """cb_stage_body: the YOLO-style stage body (1x1 C->C/2, 3x3 C/2->C/2, 1x1 on the concat + x1)
    in one kernel, C = 16 or 32.  layers: three objects with HOST float32 arrays .w_host (OHWI),
    .scale_host, .bias_host (ConvBnAct layers keep them): the call reads them and puts them in the
    launch."""
    xv, yv = nhwc(x1), nhwc(y)
    arrs = []
    for L in layers:
        for a in (L.w_host, L.scale_host, L.bias_host):
            a = np.ascontiguousarray(a, dtype=np.float32)
            arrs.append(a)
    st = load().cb_stage_body(ctypes.byref(xv), *[a.ctypes.data for a in arrs], act, ctypes.byref(yv),
                              _stream_ptr(stream))
    _check(st, "cb_stage_body")
    return y


def dw_separable_block_fused(x, p, y) -> bool:
    """cb_dw_separable_block_fused: the block would run as one kernel."""
    xv, yv = nhwc(x), nhwc(y)
    sk = p.get("skip_w")
    return bool(load().cb_dw_separable_block_fused(ctypes.byref(xv), ctypes.byref(yv), p["pw_w"].data_ptr(),
                                                   sk.data_ptr() if sk is not None else None))


def dw_separable_block_static(x, p, stride, y, stream=None):
    """cb_dw_separable_block_static: the same block with the library's fixed scratch array
    (no workspace argument, no allocation).  Returns the cb status without raising."""
    xv, yv = nhwc(x), nhwc(y)
    sk = p.get("skip_w")
    return load().cb_dw_separable_block_static(
        ctypes.byref(xv), p["dw_w"].data_ptr(), p["dw_scale"].data_ptr(), p["dw_bias"].data_ptr(),
        p["pw_w"].data_ptr(), p["pw_scale"].data_ptr(), p["pw_bias"].data_ptr(),
        sk.data_ptr() if sk is not None else None,
        p["skip_scale"].data_ptr() if sk is not None else None,
        p["skip_bias"].data_ptr() if sk is not None else None,
        stride, ctypes.byref(yv), _stream_ptr(stream))


def avgpool_linear(x, fc_w, fc_b, out, stream=None):
    xv = nhwc(x)
    _check(load().cb_avgpool_linear(ctypes.byref(xv), fc_w.data_ptr(), fc_b.data_ptr(), fc_w.shape[0],
                                    out.data_ptr(), _stream_ptr(stream)), "cb_avgpool_linear")
    return out


def preprocess_u8(src, dst, stream=None):
    """src: uint8 [N, Hs, Ws, 3] device tensor (rows may be padded: src.stride(1) is the pitch);
    dst: float32 [N, 3, Hd, Wd] contiguous device tensor."""
    N, Hs, Ws, _ = src.shape
    _, _, Hd, Wd = dst.shape
    assert src.stride(0) == Hs * src.stride(1) and src.stride(2) == 3 and src.stride(3) == 1
    _check(load().cb_preprocess_u8(src.data_ptr(), N, Hs, Ws, src.stride(1), dst.data_ptr(), Hd, Wd,
                                   _stream_ptr(stream)), "cb_preprocess_u8")
    return dst


def preprocess_stem_u8(src, dst_hw, w, scale, bias, act, y, stream=None):
    """cb_preprocess_stem_u8: u8 frames [N, Hs, Ws, 3] (rows may be padded) resized to dst_hw, /255,
    straight into the 3 -> 16 stride-2 stem; y: [N, OH, OW, 16] NHWC view; w, scale, bias: device
    tensors in the cb_repack_weights / cb_fold_bn layouts."""
    N, Hs, Ws, _ = src.shape
    assert src.stride(0) == Hs * src.stride(1) and src.stride(2) == 3 and src.stride(3) == 1
    yv = nhwc(y)
    _check(load().cb_preprocess_stem_u8(src.data_ptr(), N, Hs, Ws, src.stride(1), dst_hw[0], dst_hw[1],
                                        w.data_ptr(), scale.data_ptr(), bias.data_ptr(), act, ctypes.byref(yv),
                                        _stream_ptr(stream)), "cb_preprocess_stem_u8")
    return y


def preprocess_u8_three_pass(src, tmp_u8, tmp_f32, dst, stream=None):
    N, Hs, Ws, _ = src.shape
    _, _, Hd, Wd = dst.shape
    _check(load().cb_preprocess_u8_three_pass(src.data_ptr(), N, Hs, Ws, src.stride(1), tmp_u8.data_ptr(),
                                              tmp_f32.data_ptr(), dst.data_ptr(), Hd, Wd, _stream_ptr(stream)),
           "cb_preprocess_u8_three_pass")
    return dst


def debug_timeout_probe(timeout_ms, stream=None):
    """cb_debug_timeout_probe: a bounded wait that nothing satisfies (tests the timeout report)."""
    _check(load().cb_debug_timeout_probe(int(timeout_ms), _stream_ptr(stream)), "cb_debug_timeout_probe")


def debug_sample_coords(src_extent, dst_extent, device="cuda", stream=None):
    """cb_debug_sample_coords: the (i0, i1, frac) the preprocess kernels use along one axis, as numpy."""
    import torch
    i0 = torch.empty(dst_extent, dtype=torch.int32, device=device)
    i1 = torch.empty(dst_extent, dtype=torch.int32, device=device)
    a = torch.empty(dst_extent, dtype=torch.float32, device=device)
    _check(load().cb_debug_sample_coords(int(src_extent), int(dst_extent), i0.data_ptr(), i1.data_ptr(),
                                         a.data_ptr(), _stream_ptr(stream)), "cb_debug_sample_coords")
    torch.cuda.synchronize()
    return i0.cpu().numpy(), i1.cpu().numpy(), a.cpu().numpy()


def get_device_error(stream=None) -> int:
    return load().cb_get_device_error(_stream_ptr(stream))
