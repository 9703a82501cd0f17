"""GPU parity of cb_stage_body: the body of a YOLO-style stage (1x1 C->C/2, 3x3 C/2->C/2 on its
output, 1x1 on the concat [a | b] with x1 added after the activation) in one kernel.

C = 16 (stage 0 of the chain):

The kernel computes in fp32 on the CUDA cores and keeps a and b in shared memory: the bar is the
fp32 one (1e-5 of max|oracle|) against the oracle's three layers composed.  Shapes cover one and
several 4 x 32 output tiles, ragged tile edges in both directions and images smaller than a tile
(the 3x3's zero padding sits inside the tile there); the three activations; a channel-slice input
and an output slice with canaries around it; bf16 storage (within half a bf16 ulp of the oracle on
the same bf16 values, and bit-equal to the fp32 kernel's output rounded); the three-layer path;
and the argument checks.

C = 32 (stage 1) runs on the tensor cores with TF32 operands, the precision of the tensor-core
layers: the bar is the TF32 one (5e-3 of max|oracle|), every output is a TF32 value (the low 13
mantissa bits clear), and the shapes add one with more tiles than the grid has warpgroups, so that
each warpgroup walks several tiles (the next tile's copy issued early, the output store of one tile
in flight while the next is computed).  With bf16 storage it stores a and b as bf16 (nearest even),
as the three layers store them, multiplies the 3x3's weights as bf16 like the bf16 tensor-core
layer, and the 1x1 layers' weights split into a bf16 head and tail (fp32 accuracy, as the CUDA-core
1x1 layers): held to the bf16 bar (5e-3 of max|oracle|) against the oracle composed with the same
storage (a, b and the 3x3's weights rounded to bf16), and to twice that against the oracle without
it (measured: bf16 storage of a and b alone moves the output by up to 3.6e-3).
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct
from gpu_util import TOL_BF16, TOL_FP32, TOL_TF32, bf16_within_half_ulp, canary_buffer, canary_buffer_bf16, is_canary, \
    is_canary_bf16, oracle_stage_body, oracle_stage_body_bf16_storage, rel_err, sync_check, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

SHAPES = [(2, 20, 40), (1, 16, 32), (3, 17, 33), (1, 1, 1), (1, 2, 3), (2, 40, 70), (1, 33, 95), (1, 48, 8)]


def _stage(seed, C=16):
    """A stage body's parameters with C channels (stage 0 of the chain: 16, stage 1: 32), reseeded."""
    g = np.random.default_rng(seed)
    st = {}
    h = C // 2
    for key, (co, ci, k) in {"cv1": (h, C, 1), "cv2": (h, h, 3), "cv3": (C, C, 1)}.items():
        st[key + "_w"] = synthetic.kaiming(g, co, ci, k, k)
        st[key + "_bn"] = synthetic.bn_params(g, co)
    return st


def _layers(st, act, dtype=torch.float32):
    return (ConvBnAct(st["cv1_w"], st["cv1_bn"], 1, 0, act, dtype=dtype),
            ConvBnAct(st["cv2_w"], st["cv2_bn"], 1, 1, act, dtype=dtype),
            ConvBnAct(st["cv3_w"], st["cv3_bn"], 1, 0, act, dtype=dtype))


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stage_body_silu(gpu, orc, shape):
    N, H, W = shape
    st = _stage(N + H + W)
    x1 = np.random.default_rng(H * W).standard_normal((N, H, W, 16)).astype(np.float32)
    y = torch.empty(N, H, W, 16, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    assert "stage_body_kernel" in cb.last_launch()["kernel"]
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_FP32


@pytest.mark.parametrize("act", [cb.ACT_NONE, cb.ACT_RELU])
def test_stage_body_activations(gpu, orc, act):
    N, H, W = 2, 18, 36
    st = _stage(act + 40)
    x1 = np.random.default_rng(act).standard_normal((N, H, W, 16)).astype(np.float32)
    y = torch.empty(N, H, W, 16, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, act), act, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st, act=act)) <= TOL_FP32


def test_stage_body_matches_the_three_layers(gpu, orc):
    """The fused body against the same body run as three cb_conv_bn_act calls (the pointwise and
    8-channel 3x3 kernels, a and b through memory): both fp32, both within the fp32 bar."""
    N, H, W = 4, 50, 64
    st = _stage(7)
    x1 = np.random.default_rng(7).standard_normal((N, H, W, 16)).astype(np.float32)
    l1, l2, l3 = _layers(st, cb.ACT_SILU)
    xd = to_dev(x1)
    y = torch.empty(N, H, W, 16, device=gpu)
    cb.stage_body(xd, (l1, l2, l3), cb.ACT_SILU, y)
    cat = torch.empty(N, H, W, 16, device=gpu)
    y3 = torch.empty_like(y)
    l1(xd, cat[..., :8])
    l2(cat[..., :8], cat[..., 8:])
    l3(cat, y3, residual=xd, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = oracle_stage_body(orc, x1, st)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32
    assert rel_err(y.cpu().numpy(), y3.cpu().numpy()) <= 2 * TOL_FP32


def test_stage_body_views(gpu, orc):
    """x1 as channels [8, 24) of a 32-channel buffer; the output into channels [16, 32) of a
    40-channel buffer with padded rows: nothing around it is written."""
    N, H, W = 2, 19, 45
    st = _stage(3)
    wide = np.random.default_rng(3).standard_normal((N, H, W, 32)).astype(np.float32)
    x1 = np.ascontiguousarray(wide[..., 8:24])
    xd = to_dev(wide)[..., 8:24]
    buf = canary_buffer((N, H, W + 5, 40))
    y = buf[:, :, :W, 16:32]
    cb.stage_body(xd, _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_FP32
    assert is_canary(buf[..., :16]) and is_canary(buf[..., 32:]) and is_canary(buf[:, :, W:])


@pytest.mark.parametrize("shape", [(2, 20, 40), (3, 17, 33), (1, 2, 3), (2, 40, 70)],
                         ids=lambda s: "x".join(map(str, s)))
def test_stage_body_bf16(gpu, orc, shape):
    """bf16 storage: x1 read and the output written as bfloat16, the weights and every product and
    sum in fp32 (a and b stay fp32 in shared memory)."""
    N, H, W = shape
    st = _stage(N * H + W)
    x1 = np.random.default_rng(W).standard_normal((N, H, W, 16)).astype(np.float32)
    xd, xv = to_dev_bf16(x1)
    buf = canary_buffer_bf16((N, H, W, 32))
    y = buf[..., 8:24]  # 16-byte aligned channel slice
    cb.stage_body(xd, _layers(st, cb.ACT_SILU, dtype=torch.bfloat16), cb.ACT_SILU, y)
    sync_check()
    ref = oracle_stage_body(orc, xv, st)
    got = y.float().cpu().numpy()
    assert bf16_within_half_ulp(got, ref) <= 1.0
    assert is_canary_bf16(buf[..., :8]) and is_canary_bf16(buf[..., 24:])
    y32 = torch.empty(N, H, W, 16, device=gpu)
    cb.stage_body(torch.from_numpy(xv).to(gpu), _layers(st, cb.ACT_SILU), cb.ACT_SILU, y32)
    sync_check()
    assert torch.equal(y.contiguous().view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))


def test_stage_body_full_size_stage0(gpu, orc):
    """The chain's stage 0 body at its size (320 x 320, batch 32, the 640 x 640 input's stride-2
    output), every output against the oracle."""
    stages = synthetic.yolo_params()
    st = stages[0]
    x1 = np.random.default_rng(5).standard_normal((32, 320, 320, 16)).astype(np.float32)
    y = torch.empty(32, 320, 320, 16, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_FP32


def test_stage_body_rejects(gpu):
    st = _stage(1)
    layers = _layers(st, cb.ACT_SILU)
    x1 = torch.zeros(1, 8, 8, 16, device=gpu)
    with pytest.raises(cb.CbError) as e:  # in place: the output overlaps x1
        cb.stage_body(x1, layers, cb.ACT_SILU, x1)
    assert e.value.status == cb.ERR_INVALID_ARG
    with pytest.raises(cb.CbError) as e:  # shape mismatch
        cb.stage_body(x1, layers, cb.ACT_SILU, torch.empty(1, 8, 7, 16, device=gpu))
    assert e.value.status == cb.ERR_INVALID_ARG
    with pytest.raises(cb.CbError) as e:  # dtype mismatch
        cb.stage_body(x1, layers, cb.ACT_SILU, torch.empty(1, 8, 8, 16, device=gpu, dtype=torch.bfloat16))
    assert e.value.status == cb.ERR_INVALID_ARG
    with pytest.raises(cb.CbError) as e:  # 8 channels: no kernel
        cb.stage_body(torch.zeros(1, 8, 8, 8, device=gpu), layers, cb.ACT_SILU, torch.empty(1, 8, 8, 8, device=gpu))
    assert e.value.status == cb.ERR_UNSUPPORTED
    with pytest.raises(cb.CbError) as e:  # pixels 18 floats apart: not whole 16-byte pieces
        cb.stage_body(torch.zeros(1, 8, 8, 18, device=gpu)[..., :16], layers, cb.ACT_SILU,
                      torch.empty(1, 8, 8, 16, device=gpu))
    assert e.value.status == cb.ERR_ALIGNMENT


# ----------------------------------------------------------------- C = 32: tensor cores
SHAPES32 = [(2, 20, 40), (1, 4, 32), (3, 17, 33), (1, 1, 1), (1, 2, 3), (2, 40, 70), (1, 33, 95), (1, 48, 8),
            (8, 102, 130)]


def _is_tf32(t):
    return bool(((t.contiguous().view(torch.int32) & 0x1FFF) == 0).all().item())


@pytest.mark.parametrize("shape", SHAPES32, ids=lambda s: "x".join(map(str, s)))
def test_stage_body_c32(gpu, orc, shape):
    N, H, W = shape
    st = _stage(N + H + W, C=32)
    x1 = np.random.default_rng(H * W + 1).standard_normal((N, H, W, 32)).astype(np.float32)
    y = torch.empty(N, H, W, 32, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    assert "stage_body_tc_kernel" in cb.last_launch()["kernel"]
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_TF32
    assert _is_tf32(y)


@pytest.mark.parametrize("act", [cb.ACT_NONE, cb.ACT_RELU])
def test_stage_body_c32_activations(gpu, orc, act):
    N, H, W = 2, 18, 36
    st = _stage(act + 60, C=32)
    x1 = np.random.default_rng(act + 9).standard_normal((N, H, W, 32)).astype(np.float32)
    y = torch.empty(N, H, W, 32, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, act), act, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st, act=act)) <= TOL_TF32


def test_stage_body_c32_matches_the_three_layers(gpu, orc):
    """The fused body against the same body run as three cb_conv_bn_act calls (a and b through
    memory): both within the TF32 bar of the oracle and of each other."""
    N, H, W = 4, 50, 64
    st = _stage(8, C=32)
    x1 = np.random.default_rng(8).standard_normal((N, H, W, 32)).astype(np.float32)
    l1, l2, l3 = _layers(st, cb.ACT_SILU)
    xd = to_dev(x1)
    y = torch.empty(N, H, W, 32, device=gpu)
    cb.stage_body(xd, (l1, l2, l3), cb.ACT_SILU, y)
    cat = torch.empty(N, H, W, 32, device=gpu)
    y3 = torch.empty_like(y)
    l1(xd, cat[..., :16])
    l2(cat[..., :16], cat[..., 16:])
    l3(cat, y3, residual=xd, res_mode=cb.RES_POST_ACT)
    sync_check()
    ref = oracle_stage_body(orc, x1, st)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_TF32
    assert rel_err(y.cpu().numpy(), y3.cpu().numpy()) <= 2 * TOL_TF32


def test_stage_body_c32_views(gpu, orc):
    """x1 as channels [16, 48) of a 64-channel buffer; the output into channels [4, 36) of a
    40-channel buffer with padded rows: the tensor store writes nothing around it."""
    N, H, W = 2, 19, 45
    st = _stage(4, C=32)
    wide = np.random.default_rng(4).standard_normal((N, H, W, 64)).astype(np.float32)
    x1 = np.ascontiguousarray(wide[..., 16:48])
    xd = to_dev(wide)[..., 16:48]
    buf = canary_buffer((N, H, W + 5, 40))
    y = buf[:, :, :W, 4:36]
    cb.stage_body(xd, _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_TF32
    assert is_canary(buf[..., :4]) and is_canary(buf[..., 36:]) and is_canary(buf[:, :, W:])


def test_stage_body_c32_full_size_stage1(gpu, orc):
    """The chain's stage 1 body at its size (160 x 160, batch 32, the 640 x 640 input's second
    stride-2 output), every output against the oracle."""
    st = synthetic.yolo_params()[1]
    x1 = np.random.default_rng(6).standard_normal((32, 160, 160, 32)).astype(np.float32)
    y = torch.empty(32, 160, 160, 32, device=gpu)
    cb.stage_body(to_dev(x1), _layers(st, cb.ACT_SILU), cb.ACT_SILU, y)
    sync_check()
    assert rel_err(y.cpu().numpy(), oracle_stage_body(orc, x1, st)) <= TOL_TF32


def test_stage_body_c32_rejects(gpu):
    layers = _layers(_stage(2, C=32), cb.ACT_SILU)
    with pytest.raises(cb.CbError) as e:  # bf16 output pixels 36 elements (72 bytes) apart: no tensor store
        cb.stage_body(torch.zeros(1, 8, 8, 32, device=gpu, dtype=torch.bfloat16), layers, cb.ACT_SILU,
                      torch.empty(1, 8, 8, 36, device=gpu, dtype=torch.bfloat16)[..., :32])
    assert e.value.status == cb.ERR_ALIGNMENT
    with pytest.raises(cb.CbError) as e:  # 24 channels: no kernel
        cb.stage_body(torch.zeros(1, 8, 8, 24, device=gpu), layers, cb.ACT_SILU, torch.empty(1, 8, 8, 24, device=gpu))
    assert e.value.status == cb.ERR_UNSUPPORTED
    x1 = torch.zeros(1, 8, 8, 32, device=gpu)
    with pytest.raises(cb.CbError) as e:  # in place
        cb.stage_body(x1, layers, cb.ACT_SILU, x1)
    assert e.value.status == cb.ERR_INVALID_ARG
    with pytest.raises(cb.CbError) as e:  # output rows 34 floats apart: not whole 16-byte pieces
        cb.stage_body(x1, layers, cb.ACT_SILU, torch.empty(1, 8, 8, 34, device=gpu)[..., :32])
    assert e.value.status == cb.ERR_ALIGNMENT


@pytest.mark.parametrize("shape", [(2, 20, 40), (1, 1, 1), (3, 17, 33), (1, 33, 95), (8, 102, 130)],
                         ids=lambda s: "x".join(map(str, s)))
def test_stage_body_c32_bf16(gpu, orc, shape):
    """bf16 storage: x1 read and the output written as bfloat16 by the tensor-core body (bf16
    operands, fp32 accumulate), against the oracle on the same bf16 x1; a channel slice of a wider
    output buffer with canaries around it."""
    N, H, W = shape
    st = _stage(N * W + 5, C=32)
    x1 = np.random.default_rng(H + 3).standard_normal((N, H, W, 32)).astype(np.float32)
    xd, xv = to_dev_bf16(x1)
    buf = canary_buffer_bf16((N, H, W, 48))
    y = buf[..., 8:40]  # 16-byte aligned channel slice, pixels 96 bytes apart
    cb.stage_body(xd, _layers(st, cb.ACT_SILU, dtype=torch.bfloat16), cb.ACT_SILU, y)
    assert "stage_body_tc_kernel" in cb.last_launch()["kernel"]
    sync_check()
    got = y.float().cpu().numpy()
    assert rel_err(got, oracle_stage_body_bf16_storage(orc, xv, st)) <= TOL_BF16
    assert rel_err(got, oracle_stage_body(orc, xv, st)) <= 2 * TOL_BF16
    assert is_canary_bf16(buf[..., :8]) and is_canary_bf16(buf[..., 40:])


def test_stage_body_c32_bf16_full_size_stage1(gpu, orc):
    """The bf16 chain's stage 1 body at its size (160 x 160, batch 32), every output."""
    st = synthetic.yolo_params()[1]
    x1 = np.random.default_rng(9).standard_normal((32, 160, 160, 32)).astype(np.float32)
    xd, xv = to_dev_bf16(x1)
    y = torch.empty(32, 160, 160, 32, device=gpu, dtype=torch.bfloat16)
    cb.stage_body(xd, _layers(st, cb.ACT_SILU, dtype=torch.bfloat16), cb.ACT_SILU, y)
    sync_check()
    got = y.float().cpu().numpy()
    assert rel_err(got, oracle_stage_body_bf16_storage(orc, xv, st)) <= TOL_BF16
    assert rel_err(got, oracle_stage_body(orc, xv, st)) <= 2 * TOL_BF16


@pytest.mark.parametrize("act", [cb.ACT_NONE, cb.ACT_RELU])
def test_stage_body_c32_bf16_activations(gpu, orc, act):
    N, H, W = 2, 18, 36
    st = _stage(act + 80, C=32)
    x1 = np.random.default_rng(act + 19).standard_normal((N, H, W, 32)).astype(np.float32)
    xd, xv = to_dev_bf16(x1)
    y = torch.empty(N, H, W, 32, device=gpu, dtype=torch.bfloat16)
    cb.stage_body(xd, _layers(st, act, dtype=torch.bfloat16), act, y)
    sync_check()
    got = y.float().cpu().numpy()
    assert rel_err(got, oracle_stage_body_bf16_storage(orc, xv, st, act=act)) <= TOL_BF16
    assert rel_err(got, oracle_stage_body(orc, xv, st, act=act)) <= 2 * TOL_BF16


@pytest.mark.parametrize("C,dtype", [(16, torch.float32), (32, torch.float32), (32, torch.bfloat16)],
                         ids=["c16_fp32", "c32_fp32", "c32_bf16"])
def test_stage_body_nan_propagates(gpu, orc, C, dtype):
    """A NaN in x1 reaches exactly the outputs the oracle makes NaN -- the pixel's 3x3 neighbourhood
    (through b) -- and no rounding or masking step turns it into a number; every other output
    still meets the bar."""
    N, H, W = 1, 12, 40
    st = _stage(C + 5, C=C)
    x1 = np.random.default_rng(C).standard_normal((N, H, W, C)).astype(np.float32)
    x1[0, 5, 17, 3] = np.nan
    if dtype == torch.bfloat16:
        xd, xv = to_dev_bf16(x1)
    else:
        xd, xv = to_dev(x1), x1
    y = torch.empty(N, H, W, C, device=gpu, dtype=dtype)
    cb.stage_body(xd, _layers(st, cb.ACT_SILU, dtype=dtype), cb.ACT_SILU, y)
    sync_check()
    got = y.float().cpu().numpy()
    ref = oracle_stage_body(orc, xv, st)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(ref[0, 4:7, 16:19]).all() and not np.isnan(ref[0, 8:, :]).any()
    fin = ~np.isnan(ref)
    tol = TOL_FP32 if C == 16 else (TOL_TF32 if dtype == torch.float32 else 2 * TOL_BF16)
    assert np.max(np.abs(got[fin] - ref[fin])) <= tol * np.max(np.abs(ref[fin]))
