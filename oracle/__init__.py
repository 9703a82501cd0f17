"""Plain CPU oracle (fp64) for the fused conv + BatchNorm + activation path.

TEST INFRASTRUCTURE ONLY.  The product library never imports this package;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may.  It shares no code with the CUDA path: the arithmetic lives
in ``oracle.c`` (plain C, compiled with gcc) and the compositions below chain
those primitives in the order the pages give them.

Sources (page title, section):
  * "How I sped up convolutions" -- DepthwiseSeparableConv / DepthwiseMNIST
    class listings (block and model structure) and the Metal kernel
    walk-through, steps 1-5 (window origin, zero padding, unfolded BN, ReLU).
  * "YOLO26N Inference Optimisation" -- fused conv + BN + SiLU, residual add
    and channel concat as separate passes (nsys breakdown; improvements #6, #7).
  * "A fused Ampere preprocess kernel" -- the byte ledger (resize, normalize,
    layout) and "bilinear is a contract" (OpenCV half-pixel convention).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

NHWC, NCHW = 0, 1
ACT_NONE, ACT_RELU, ACT_SILU = 0, 1, 2
RES_NONE, RES_PRE_ACT, RES_POST_ACT = 0, 1, 2
PREC_F64, PREC_F32 = 64, 32
BN_EPS = 1e-5

_F = ctypes.POINTER(ctypes.c_float)
_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I = ctypes.POINTER(ctypes.c_int)
_LL = ctypes.POINTER(ctypes.c_longlong)


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FP contraction)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.orc_out_size.restype = ctypes.c_int
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_conv2d.restype = None
        lib.orc_conv_bn_act.restype = None
        lib.orc_conv_bn_act_points.restype = None
        _lib = lib
    return _lib


def _fp(a):
    return a.ctypes.data_as(_F)


def _dp(a):
    return a.ctypes.data_as(_D)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def num_threads() -> int:
    return int(_load().orc_num_threads())


def set_num_threads(n: int) -> None:
    _load().orc_set_num_threads(ctypes.c_int(n))


def out_size(n: int, k: int, s: int, p: int) -> int:
    return (n + 2 * p - k) // s + 1


# --------------------------------------------------------------------------
# Convolution layer
# --------------------------------------------------------------------------
def _x_dims(x, layout):
    if layout == NHWC:
        N, H, W, C = x.shape
    else:
        N, C, H, W = x.shape
    return N, C, H, W


def conv2d(x, w_oihw, stride=1, pad=0, groups=1, layout=NHWC):
    """Raw convolution (no BN), fp64 NHWC output [N, OH, OW, Co]."""
    x, w = _f32(x), _f32(w_oihw)
    N, C, H, W = _x_dims(x, layout)
    Co, cin_g, kh, kw = w.shape
    assert C == cin_g * groups and Co % groups == 0
    OH, OW = out_size(H, kh, stride, pad), out_size(W, kw, stride, pad)
    z = np.empty((N, OH, OW, Co), dtype=np.float64)
    _load().orc_conv2d(_fp(x), layout, N, C, H, W, _fp(w), Co, kh, kw, stride, pad, groups, _dp(z))
    return z


def batchnorm(z, gamma, beta, mean, var, eps=BN_EPS):
    """Unfolded inference BatchNorm over the last (channel) axis, fp64."""
    z = np.ascontiguousarray(z, dtype=np.float64).copy()
    C = z.shape[-1]
    g, b, m, v = (_f32(t) for t in (gamma, beta, mean, var))
    _load().orc_batchnorm(_dp(z), ctypes.c_longlong(z.size // C), C, _fp(g), _fp(b), _fp(m), _fp(v),
                          ctypes.c_double(eps))
    return z


def activation(v, act):
    v = np.ascontiguousarray(v, dtype=np.float64).copy()
    _load().orc_activation(_dp(v), ctypes.c_longlong(v.size), act)
    return v


def conv_bn_act(x, w_oihw, bn, stride=1, pad=0, groups=1, act=ACT_NONE, residual=None,
                res_mode=RES_NONE, layout=NHWC, eps=BN_EPS):
    """The fused layer: conv -> BN (unfolded) -> residual/activation.  fp64 NHWC out.

    bn = (gamma, beta, mean, var).  residual: NHWC array of the output's shape.
    """
    x, w = _f32(x), _f32(w_oihw)
    N, C, H, W = _x_dims(x, layout)
    Co, cin_g, kh, kw = w.shape
    assert C == cin_g * groups
    OH, OW = out_size(H, kh, stride, pad), out_size(W, kw, stride, pad)
    g, b, m, v = (_f32(t) for t in bn)
    y = np.empty((N, OH, OW, Co), dtype=np.float64)
    if res_mode != RES_NONE:
        r = _f32(residual)
        assert r.shape == y.shape
        rp = _fp(r)
    else:
        rp = None
    _load().orc_conv_bn_act(_fp(x), layout, N, C, H, W, _fp(w), Co, kh, kw, stride, pad, groups,
                            _fp(g), _fp(b), _fp(m), _fp(v), ctypes.c_double(eps), act, rp, res_mode,
                            _dp(y))
    return y


def conv_bn_act_points(x, w_oihw, bn, flat_idx, stride=1, pad=0, groups=1, act=ACT_NONE,
                       residual=None, res_mode=RES_NONE, layout=NHWC, eps=BN_EPS):
    """The fused layer evaluated only at flat NHWC output indices ``flat_idx``."""
    x, w = _f32(x), _f32(w_oihw)
    N, C, H, W = _x_dims(x, layout)
    Co, cin_g, kh, kw = w.shape
    g, b, m, v = (_f32(t) for t in bn)
    idx = np.ascontiguousarray(flat_idx, dtype=np.int64)
    out = np.empty(idx.shape, dtype=np.float64)
    rp = None
    if res_mode != RES_NONE:
        keep = _f32(residual).reshape(-1)
        rp = _fp(keep)
    _load().orc_conv_bn_act_points(_fp(x), layout, N, C, H, W, _fp(w), Co, kh, kw, stride, pad,
                                   groups, _fp(g), _fp(b), _fp(m), _fp(v), ctypes.c_double(eps), act,
                                   rp, res_mode, idx.ctypes.data_as(_LL), ctypes.c_longlong(idx.size),
                                   _dp(out))
    return out


def global_avgpool(x):
    """AdaptiveAvgPool2d(1) over an NHWC fp64 tensor -> [N, C]."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    N, H, W, C = x.shape
    out = np.empty((N, C), dtype=np.float64)
    _load().orc_global_avgpool(_dp(x), N, H, W, C, _dp(out))
    return out


def linear(x, w, b):
    x = np.ascontiguousarray(x, dtype=np.float64)
    w, b = _f32(w), _f32(b)
    N, In = x.shape
    Out = w.shape[0]
    out = np.empty((N, Out), dtype=np.float64)
    _load().orc_linear(_dp(x), N, In, _fp(w), _fp(b), Out, _dp(out))
    return out


# --------------------------------------------------------------------------
# Blocks and models ("How I sped up convolutions", class listings)
# --------------------------------------------------------------------------
def dw_separable_block(x, p, stride):
    """DepthwiseSeparableConv.forward on an NHWC fp32 input; fp64 NHWC out.

    p: dict with 'dw_w' [Cin,1,3,3], 'bn1', 'pw_w' [Cout,Cin,1,1], 'bn2' and,
    when stride != 1 or Cin != Cout, 'skip_w' [Cout,Cin,1,1] and 'skip_bn'.
    Steps, in the listing's order: t = relu(bn1(dw3x3_s(x)));
    u = bn2(pw(t)); identity = skip(x) or x; out = relu(u + identity).
    The workload is an fp32 network, so the stored activation t is fp32; all
    arithmetic inside each step is fp64.
    """
    Cin = x.shape[-1]
    Cout = p["pw_w"].shape[0]
    t = conv_bn_act(x, p["dw_w"], p["bn1"], stride=stride, pad=1, groups=Cin, act=ACT_RELU)
    t = t.astype(np.float32)
    u = batchnorm(conv2d(t, p["pw_w"]), *p["bn2"])
    if stride != 1 or Cin != Cout:
        ident = batchnorm(conv2d(x, p["skip_w"], stride=stride), *p["skip_bn"])
    else:
        ident = np.asarray(x, dtype=np.float64)
    return activation(u + ident, ACT_RELU)


def mnist_model(x, params):
    """DepthwiseMNIST forward on NHWC fp32 input [N, 28, 28, 1] -> logits [N, 10] (fp64)."""
    h = conv_bn_act(x, params["stem_w"], params["stem_bn"], stride=1, pad=1, act=ACT_RELU)
    for blk, (cin, cout, s) in zip(params["blocks"], MNIST_BLOCKS):
        h = dw_separable_block(h.astype(np.float32), blk, s)
    pooled = global_avgpool(h)
    return linear(pooled, params["fc_w"], params["fc_b"])


MNIST_BLOCKS = ((48, 96, 2), (96, 96, 1), (96, 192, 2), (192, 192, 1))


def mnist_param_count(params) -> int:
    """Conv weights + BN affine (gamma, beta) + fc weight and bias."""
    total = params["stem_w"].size + 2 * params["stem_bn"][0].size
    for blk in params["blocks"]:
        total += blk["dw_w"].size + 2 * blk["bn1"][0].size
        total += blk["pw_w"].size + 2 * blk["bn2"][0].size
        if "skip_w" in blk:
            total += blk["skip_w"].size + 2 * blk["skip_bn"][0].size
    return int(total + params["fc_w"].size + params["fc_b"].size)


def yolo_stage(x, stage):
    """One stage of the YOLO-style chain on NHWC fp32 input; fp64 NHWC out.

    x1 = silu(bn(conv3x3 s2(x)));  a = silu(bn(conv1x1(x1)))  (C -> C/2);
    b = silu(bn(conv3x3(a)))  (C/2 -> C/2);  cat = [a | b]  (a first);
    out = silu(bn(conv1x1(cat))) + x1  (post-activation residual).
    """
    x1 = conv_bn_act(x, stage["down_w"], stage["down_bn"], stride=2, pad=1, act=ACT_SILU)
    x1f = x1.astype(np.float32)
    a = conv_bn_act(x1f, stage["cv1_w"], stage["cv1_bn"], act=ACT_SILU)
    af = a.astype(np.float32)
    b = conv_bn_act(af, stage["cv2_w"], stage["cv2_bn"], pad=1, act=ACT_SILU)
    cat = np.concatenate([af, b.astype(np.float32)], axis=-1)
    return conv_bn_act(cat, stage["cv3_w"], stage["cv3_bn"], act=ACT_SILU, residual=x1f,
                       res_mode=RES_POST_ACT)


# --------------------------------------------------------------------------
# Preprocess ("A fused Ampere preprocess kernel")
# --------------------------------------------------------------------------
def axis_coords(S, D, prec=PREC_F64):
    i0 = np.empty(D, dtype=np.int32)
    i1 = np.empty(D, dtype=np.int32)
    a = np.empty(D, dtype=np.float64)
    _load().orc_axis_coords(S, D, prec, i0.ctypes.data_as(_I), i1.ctypes.data_as(_I), _dp(a))
    return i0, i1, a


def _src_args(src):
    src = np.ascontiguousarray(src, dtype=np.uint8)
    N, Hs, Ws, C = src.shape
    assert C == 3
    return src, N, Hs, Ws, Ws * 3


def resize_u8(src, Hd, Wd, prec=PREC_F64, return_values=False):
    """Pass 1: bilinear resize, rounded half up to u8, HWC out [N, Hd, Wd, 3]."""
    src, N, Hs, Ws, pitch = _src_args(src)
    out = np.empty((N, Hd, Wd, 3), dtype=np.uint8)
    v = np.empty((N, Hd, Wd, 3), dtype=np.float64) if return_values else None
    _load().orc_resize_u8(src.ctypes.data_as(_U8), N, Hs, Ws, ctypes.c_longlong(pitch), Hd, Wd, prec,
                          out.ctypes.data_as(_U8), _dp(v) if v is not None else None)
    return (out, v) if return_values else out


def normalize_u8(u):
    """Pass 2: u8 -> fp32 u / 255 (one IEEE fp32 division)."""
    u = np.ascontiguousarray(u, dtype=np.uint8)
    out = np.empty(u.shape, dtype=np.float32)
    _load().orc_normalize_u8(u.ctypes.data_as(_U8), ctypes.c_longlong(u.size), _fp(out))
    return out


def hwc_to_chw(f):
    """Pass 3: fp32 [N, H, W, 3] -> [N, 3, H, W]."""
    f = _f32(f)
    N, H, W, _ = f.shape
    out = np.empty((N, 3, H, W), dtype=np.float32)
    _load().orc_hwc_to_chw(_fp(f), N, H, W, _fp(out))
    return out


def preprocess_u8(src, Hd, Wd, prec=PREC_F64):
    """Fused preprocess: u8 HWC frames -> fp32 NCHW [N, 3, Hd, Wd]."""
    src, N, Hs, Ws, pitch = _src_args(src)
    out = np.empty((N, 3, Hd, Wd), dtype=np.float32)
    _load().orc_preprocess_u8(src.ctypes.data_as(_U8), N, Hs, Ws, ctypes.c_longlong(pitch), Hd, Wd,
                              prec, _fp(out))
    return out


def preprocess_u8_three_pass(src, Hd, Wd, prec=PREC_F64):
    """The unfused pipeline: resize (u8) -> normalize (fp32 HWC) -> layout (CHW)."""
    return hwc_to_chw(normalize_u8(resize_u8(src, Hd, Wd, prec)))
