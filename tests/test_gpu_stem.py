"""GPU parity of the 3 -> 16 channel stride-2 stem kernels and of the preprocess fused into it.

Two kernels take the stem: on CUDA cores in fp32 (planar NCHW input -- the preprocess output --
and, on request, packed NHWC), and on the tensor cores with each fp32 operand split into a TF32
head and tail (packed NHWC input, the default there).  Both are held to the fp32 bar (1e-5 of
max|oracle|); every NHWC case runs on both, and the test checks which kernel launched.  Shapes
cover one and several output tiles (8 x 64 on CUDA cores, 2 x 64 on the tensor cores), ragged tile
edges in both directions, tiny images, the epilogue variants, residuals and output views with
padded rows.  The fused preprocess + stem
kernel must produce, bit for bit, what the preprocess kernel followed by the stem kernel produce
(the planar image it keeps in shared memory holds the preprocess's values and the convolution
code is shared), and match the oracle's preprocess followed by the oracle's convolution.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_FP32, canary_buffer, is_canary, rel_err, sync_check, to_dev

pytestmark = pytest.mark.gpu

SHAPES = [(2, 64, 64), (1, 30, 52), (3, 17, 132), (1, 2, 4), (1, 1, 4), (2, 40, 200), (1, 33, 264)]


def _stem(seed):
    g = np.random.default_rng(seed)
    return synthetic.kaiming(g, 16, 3, 3, 3), synthetic.bn_params(g, 16)


@pytest.fixture(params=["tc", "cuda"])
def stem_kernel(request, gpu):
    """The kernel packed NHWC stems take (CB_STEM_KERNEL); planar input always takes the CUDA-core one."""
    with cb.tuning("CB_STEM_KERNEL", request.param):
        yield request.param


def _check_kernel(kernel, layout=cb.LAYOUT_NHWC):
    name = cb.last_launch()["kernel"]
    assert "stem" in name, name
    assert ("stem_tc_kernel" in name) == (kernel == "tc" and layout == cb.LAYOUT_NHWC), name


def _run(x_dev, layer, OH, OW, layout, y=None, residual=None, res_mode=0, kernel=None):
    N = x_dev.shape[0]
    if y is None:
        y = torch.empty(N, OH, OW, 16, device="cuda")
    assert cb.conv_path(x_dev, y, 3, 2, 1, x_layout=layout) == cb.PATH_STEM
    layer(x_dev, y, residual=residual, res_mode=res_mode, x_layout=layout)
    if kernel is not None:
        _check_kernel(kernel, layout)
    sync_check()
    return y


def test_stem_nhwc_default_is_tensor_core(gpu, orc):
    """With no override, packed NHWC fp32 and bf16 stems launch the tensor-core kernel, planar ones
    the CUDA-core kernel."""
    w, bn = _stem(2)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    x = np.random.default_rng(2).standard_normal((1, 32, 64, 3)).astype(np.float32)
    _run(to_dev(x), layer, 16, 32, cb.LAYOUT_NHWC, kernel="tc")
    _run(to_dev(np.ascontiguousarray(x.transpose(0, 3, 1, 2))), layer, 16, 32, cb.LAYOUT_NCHW, kernel="tc")
    y = torch.empty(1, 16, 32, 16, dtype=torch.bfloat16, device="cuda")
    layer(to_dev(x).to(torch.bfloat16), y)
    _check_kernel("tc")
    sync_check()


@pytest.mark.parametrize("layout", ["nhwc", "nchw"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stem_silu(gpu, orc, stem_kernel, layout, shape):
    N, H, W = shape
    x = np.random.default_rng(H * W).standard_normal((N, H, W, 3)).astype(np.float32)
    w, bn = _stem(N + H)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, W)
    if layout == "nchw":
        xp = np.ascontiguousarray(x.transpose(0, 3, 1, 2))
        y = _run(to_dev(xp), layer, OH, OW, cb.LAYOUT_NCHW, kernel=stem_kernel)
        ref = orc.conv_bn_act(xp, w, bn, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
    else:
        y = _run(to_dev(x), layer, OH, OW, cb.LAYOUT_NHWC, kernel=stem_kernel)
        ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def _trunc_tf32(a):
    """a with the low 13 mantissa bits cleared: how a TF32 multiply reads an fp32 value."""
    return (np.asarray(a, np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)


@pytest.mark.parametrize("seed", [21, 22])
def test_stem_holds_fp32_bar_below_tf32_precision(gpu, orc, stem_kernel, seed):
    """Inputs 1 + u 2^-12 (u ~ U[0,1)) carry their information below TF32 precision: TF32 reads
    every one of them as 1.  A plain TF32 convolution then misses the fp32 bar by far (checked
    here with the oracle on truncated operands); both stem kernels -- the tensor-core one through
    its head / tail split of activations and weights -- meet it."""
    rng = np.random.default_rng(seed)
    N, H, W = 2, 34, 72
    x = (1.0 + rng.random((N, H, W, 3)) * 2.0**-12).astype(np.float32)
    w, bn = _stem(seed)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_NONE)
    OH, OW = layer.out_hw(H, W)
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_NONE)
    plain_tf32 = orc.conv_bn_act(_trunc_tf32(x), _trunc_tf32(w), bn, stride=2, pad=1, act=orc.ACT_NONE)
    assert rel_err(plain_tf32, ref) > 20 * TOL_FP32
    y = _run(to_dev(x), layer, OH, OW, cb.LAYOUT_NHWC, kernel=stem_kernel)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("act,res_mode", [(0, 0), (1, 0), (1, 1), (2, 2), (0, 2), (2, 1)])
def test_stem_epilogues(gpu, orc, stem_kernel, act, res_mode):
    N, H, W = 2, 26, 136
    x = np.random.default_rng(act).standard_normal((N, H, W, 3)).astype(np.float32)
    w, bn = _stem(7 + act)
    layer = ConvBnAct(w, bn, 2, 1, act)
    OH, OW = layer.out_hw(H, W)
    r = np.random.default_rng(5).standard_normal((N, OH, OW, 16)).astype(np.float32)
    y = _run(to_dev(x), layer, OH, OW, cb.LAYOUT_NHWC, residual=to_dev(r) if res_mode else None, res_mode=res_mode,
             kernel=stem_kernel)
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=act, residual=r if res_mode else None, res_mode=res_mode)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_stem_output_slice_with_padded_rows(gpu, orc, stem_kernel):
    """Output into channels [16, 32) of a 40-channel buffer with padded rows: nothing else is written."""
    N, H, W = 2, 20, 100
    x = np.random.default_rng(3).standard_normal((N, H, W, 3)).astype(np.float32)
    w, bn = _stem(3)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, W)
    buf = canary_buffer((N, OH, OW + 7, 40))
    y = buf[:, :, :OW, 16:32]
    _run(to_dev(x), layer, OH, OW, cb.LAYOUT_NHWC, y=y, kernel=stem_kernel)
    ref = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32
    assert is_canary(buf[:, :, OW:, :]) and is_canary(buf[:, :, :OW, :16]) and is_canary(buf[:, :, :OW, 32:])


def test_stem_not_taken_outside_its_shapes(gpu, orc):
    w, bn = _stem(1)
    x = torch.empty(1, 16, 33, 3, device="cuda")  # W % 4 != 0
    y = torch.empty(1, 8, 17, 16, device="cuda")
    assert cb.conv_path(x, y, 3, 2, 1) == cb.PATH_DIRECT
    x4 = torch.empty(1, 16, 32, 4, device="cuda")[..., :3]  # pixels 4 floats apart
    y = torch.empty(1, 8, 16, 16, device="cuda")
    assert cb.conv_path(x4, y, 3, 2, 1) == cb.PATH_DIRECT
    x = torch.empty(1, 16, 32, 3, device="cuda")
    assert cb.conv_path(x, torch.empty(1, 8, 16, 8, device="cuda"), 3, 2, 1) == cb.PATH_DIRECT  # Co 8
    assert cb.conv_path(x, torch.empty(1, 16, 32, 16, device="cuda"), 3, 1, 1) == cb.PATH_DIRECT  # stride 1
    cb.set_kernel_policy(1)
    try:
        assert cb.conv_path(x, y, 3, 2, 1) == cb.PATH_DIRECT
    finally:
        cb.set_kernel_policy(0)
    # an unaligned residual view takes the direct kernel, with the same result
    xa = np.random.default_rng(2).standard_normal((1, 16, 32, 3)).astype(np.float32)
    r = np.random.default_rng(3).standard_normal((1, 8, 16, 17)).astype(np.float32)
    rd = to_dev(r)[..., 1:]
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_RELU)
    yy = torch.empty(1, 8, 16, 16, device="cuda")
    layer(to_dev(xa), yy, residual=rd, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = orc.conv_bn_act(xa, w, bn, stride=2, pad=1, act=orc.ACT_RELU, residual=r[..., 1:],
                          res_mode=orc.RES_POST_ACT)
    assert rel_err(yy.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("case", ["yolo_640_b32", "yolo_640_b32_cuda", "preprocess_480x640_b32"])
def test_stem_full_size_sampled(gpu, orc, case):
    """The workloads' stems at full size, in the launch configuration the benchmark times;
    sampled outputs against the oracle point by point (first and last included)."""
    rng = np.random.default_rng(11)
    if case.startswith("yolo_640_b32"):
        x = rng.random((32, 640, 640, 3), dtype=np.float32)
        layout, okw = cb.LAYOUT_NHWC, {}
    else:
        x = np.ascontiguousarray(rng.random((32, 480, 640, 3), dtype=np.float32).transpose(0, 3, 1, 2))
        layout, okw = cb.LAYOUT_NCHW, {"layout": orc.NCHW}
    w, bn = synthetic.stem_params()
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    H, W = (x.shape[1], x.shape[2]) if layout == cb.LAYOUT_NHWC else (x.shape[2], x.shape[3])
    OH, OW = layer.out_hw(H, W)
    kernel = "cuda" if case.endswith("cuda") else "tc"
    with cb.tuning("CB_STEM_KERNEL", kernel):
        y = _run(to_dev(x), layer, OH, OW, layout, kernel=kernel)
    idx = rng.choice(y.numel(), 6000, replace=False)
    idx = np.concatenate([idx, [0, y.numel() - 1]])
    ref = orc.conv_bn_act_points(x, w, bn, idx, stride=2, pad=1, act=orc.ACT_SILU, **okw)
    got = y.reshape(-1)[torch.from_numpy(idx).to("cuda")].cpu().numpy()
    assert rel_err(got, ref) <= TOL_FP32


FUSED_SIZES = [
    # Hs, Ws, Hd, Wd: the workload ratio, exact 2:1 widths with odd heights, general ratios
    # (down and up), a ragged output tile edge
    (720, 1280, 480, 640), (16, 32, 9, 16), (45, 96, 30, 48), (100, 160, 60, 84), (30, 48, 64, 96),
    (7, 16, 13, 4), (64, 128, 64, 132),
]


def _fused(src_np, Hd, Wd, w, bn, act=cb.ACT_SILU, y=None):
    layer = ConvBnAct(w, bn, 2, 1, act)
    N = src_np.shape[0]
    OH, OW = layer.out_hw(Hd, Wd)
    if y is None:
        y = torch.empty(N, OH, OW, 16, device="cuda")
    cb.preprocess_stem_u8(to_dev(src_np), (Hd, Wd), layer.w, layer.scale, layer.bias, act, y)
    sync_check()
    return layer, y


@pytest.mark.parametrize("size", FUSED_SIZES, ids=lambda s: "%dx%d-%dx%d" % s)
def test_preprocess_stem_fused(gpu, orc, size):
    Hs, Ws, Hd, Wd = size
    N = 2
    src = synthetic.frames_u8(np.random.default_rng(Hs + Ws), (N, Hs, Ws, 3))
    w, bn = _stem(Hd)
    layer, y = _fused(src, Hd, Wd, w, bn)
    # the two-kernel path: preprocess to memory, then the stem kernel on the planar image
    planar = torch.empty(N, 3, Hd, Wd, device="cuda")
    cb.preprocess_u8(to_dev(src), planar)
    y2 = torch.empty_like(y)
    assert cb.conv_path(planar, y2, 3, 2, 1, x_layout=cb.LAYOUT_NCHW) == cb.PATH_STEM
    layer(planar, y2, x_layout=cb.LAYOUT_NCHW)
    sync_check()
    assert torch.equal(y, y2)
    ref_planar = orc.preprocess_u8(src, Hd, Wd, orc.PREC_F32)
    ref = orc.conv_bn_act(ref_planar, w, bn, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


def test_preprocess_stem_fused_view_and_relu(gpu, orc):
    N, Hs, Ws, Hd, Wd = 2, 72, 128, 48, 64
    src = synthetic.frames_u8(np.random.default_rng(4), (N, Hs, Ws, 3))
    w, bn = _stem(4)
    buf = canary_buffer((N, 24, 36, 48))
    y = buf[:, :, :32, 16:32]
    _fused(src, Hd, Wd, w, bn, act=cb.ACT_RELU, y=y)
    ref = orc.conv_bn_act(orc.preprocess_u8(src, Hd, Wd, orc.PREC_F32), w, bn, stride=2, pad=1, act=orc.ACT_RELU,
                          layout=orc.NCHW)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32
    assert is_canary(buf[:, :, 32:, :]) and is_canary(buf[:, :, :32, :16]) and is_canary(buf[:, :, :32, 32:])


def test_preprocess_stem_fused_workload_sampled(gpu, orc):
    """32 frames of the 1280x720 -> 640x480 workload: sampled outputs against the oracle chain."""
    src = synthetic.preprocess_frames(N=32)
    w, bn = synthetic.stem_params()
    _, y = _fused(src, 480, 640, w, bn)
    rng = np.random.default_rng(8)
    frames = [0, 13, 31]
    got = y.cpu().numpy()
    for f in frames:
        planar = orc.preprocess_u8(src[f:f + 1], 480, 640, orc.PREC_F32)
        idx = rng.choice(240 * 320 * 16, 1500, replace=False)
        ref = orc.conv_bn_act_points(planar, w, bn, idx, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
        assert rel_err(got[f].reshape(-1)[idx], ref) <= TOL_FP32


def test_preprocess_stem_fused_rejects(gpu):
    w, bn = _stem(1)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    src = torch.zeros(1, 16, 40, 3, dtype=torch.uint8, device="cuda")  # 120-byte rows: not a multiple of 16
    y = torch.empty(1, 4, 8, 16, device="cuda")
    with pytest.raises(cb.CbError) as e:
        cb.preprocess_stem_u8(src, (8, 16), layer.w, layer.scale, layer.bias, cb.ACT_SILU, y)
    assert e.value.status == cb.ERR_ALIGNMENT
    src = torch.zeros(1, 16, 32, 3, dtype=torch.uint8, device="cuda")
    with pytest.raises(cb.CbError) as e:  # wrong output size
        cb.preprocess_stem_u8(src, (8, 16), layer.w, layer.scale, layer.bias, cb.ACT_SILU,
                              torch.empty(1, 5, 8, 16, device="cuda"))
    assert e.value.status == cb.ERR_INVALID_ARG
    with pytest.raises(cb.CbError) as e:  # destination width not a multiple of 4
        cb.preprocess_stem_u8(src, (8, 14), layer.w, layer.scale, layer.bias, cb.ACT_SILU,
                              torch.empty(1, 4, 7, 16, device="cuda"))
    assert e.value.status == cb.ERR_ALIGNMENT


@pytest.mark.parametrize("shape", [(2, 64, 64), (1, 30, 56), (3, 17, 136), (1, 2, 8), (2, 40, 200), (1, 33, 264)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("act,res_mode", [(2, 0), (1, 1), (2, 2)])
def test_stem_bf16(gpu, orc, stem_kernel, shape, act, res_mode):
    """bf16 storage (packed NHWC bf16 input, bf16 output and residual; fp32 weights, fp32-accurate
    arithmetic): rows staged from a 16-byte boundary 8 pixels to the left of the fp32 kernel's;
    within half a bf16 ulp of the oracle on the same bf16 values, and bit-equal to the same kernel's
    fp32 output rounded (bf16 values have no TF32 tail: the fp32 tensor-core kernel's extra
    product adds zeros)."""
    from gpu_util import bf16_within_half_ulp, to_dev_bf16
    N, H, W = shape
    x = np.random.default_rng(H * W + act).standard_normal((N, H, W, 3)).astype(np.float32)
    w, bn = _stem(N + H + res_mode)
    layer = ConvBnAct(w, bn, 2, 1, act)
    OH, OW = layer.out_hw(H, W)
    r = np.random.default_rng(res_mode).standard_normal((N, OH, OW, 16)).astype(np.float32)
    xd, xv = to_dev_bf16(x)
    rd, rv = to_dev_bf16(r)
    y = torch.empty(N, OH, OW, 16, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(xd, y, 3, 2, 1) == cb.PATH_STEM
    layer(xd, y, residual=rd if res_mode else None, res_mode=res_mode)
    _check_kernel(stem_kernel)
    sync_check()
    ref = orc.conv_bn_act(xv, w, bn, stride=2, pad=1, act=act, residual=rv if res_mode else None,
                          res_mode=res_mode)
    assert bf16_within_half_ulp(y.float().cpu().numpy(), ref) <= 1.0
    y32 = torch.empty(N, OH, OW, 16, device=gpu)
    layer(torch.from_numpy(xv).to(gpu), y32, residual=torch.from_numpy(rv).to(gpu) if res_mode else None,
          res_mode=res_mode)
    sync_check()
    assert torch.equal(y.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))


def test_stem_bf16_needs_width_multiple_of_8(gpu):
    """bf16 rows are staged in 16-byte groups of 8 pixels: other widths have no bf16 stem kernel."""
    w, bn = _stem(1)
    layer = ConvBnAct(w, bn, 2, 1, cb.ACT_SILU)
    x = torch.zeros(1, 8, 12, 3, dtype=torch.bfloat16, device=gpu)
    y = torch.empty(1, 4, 6, 16, dtype=torch.bfloat16, device=gpu)
    assert cb.conv_path(x, y, 3, 2, 1) == 0
    with pytest.raises(cb.CbError) as e:
        layer(x, y)
    assert e.value.status == cb.ERR_ALIGNMENT
