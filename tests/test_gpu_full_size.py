"""Every workload checked against the oracle at its stated size, whole tensors, element by element.

The other GPU test files cover many small shapes (tiles, tails, views, epilogue variants); this
one runs each workload at the batch and image size the benchmark times, in the launch
configuration it times (the same layer objects, tile plans autotuned where the benchmark tunes),
and compares every output element with the fp64 oracle:

  * the depthwise 3x3 + BN + ReLU layer [64, 56, 56, 384] at stride 1 and 2 (fp32 bar, 1e-5);
  * each layer of the dense 3x3 + BN + SiLU sweep at batch 16 (TF32 bar on the tensor cores,
    fp32 bar on the CUDA-core stem);
  * the 20-layer YOLO-style chain at 640 x 640, batch 32 and batch 1, end to end against the
    oracle chain (5e-3: the chain holds TF32 layers), and at batch 32 layer by layer with the
    oracle fed the GPU's own input;
  * the u8 preprocess fused into the stem at batch 32 (the preprocess bit-exact, the stem 1e-5);
  * the preprocess at ratios whose weights are not dyadic, against the fp64 definition, and its
    sample coordinates against exact rational arithmetic.

Tolerance bookkeeping as everywhere: max|gpu - oracle| / max|oracle|.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import ConvBnAct, PreprocessStem, YoloChain
from gpu_util import TOL_FP32, TOL_TF32, oracle_stage_body, rel_err, stage_body_tol, sync_check, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def fresh_tuning_table():
    """These tests tune plans as the benchmark does; the table is process-wide, so it is cleared
    before and after each of them."""
    cb.autotune_clear()
    yield
    cb.autotune_clear()


def _tol(ci, co, k, stride, groups=1):
    return TOL_TF32 if cb.layer_uses_tensor_cores(ci, co, k, stride, groups) else TOL_FP32


@pytest.mark.parametrize("stride", [1, 2])
def test_depthwise_full_workload(gpu, orc, stride):
    """[64, 56, 56, 384] ~ N(0,1), w ~ N(0, 1/9): all 77 M (stride 1) or 19 M (stride 2) outputs."""
    x, w, bn = synthetic.depthwise_layer()
    layer = ConvBnAct(w, bn, stride, 1, cb.ACT_RELU, groups=384)
    OH, OW = layer.out_hw(56, 56)
    y = torch.empty(64, OH, OW, 384, device=gpu)
    assert cb.conv_path(to_dev(x), y, 3, stride, 1, groups=384) == cb.PATH_DEPTHWISE
    layer(to_dev(x), y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=stride, pad=1, groups=384, act=orc.ACT_RELU)
    assert rel_err(y.cpu().numpy(), ref) <= TOL_FP32


@pytest.mark.parametrize("layer_spec", synthetic.DENSE_SWEEP, ids=lambda s: "%d-%d@%d_s%d" % s)
def test_dense_sweep_batch16_full(gpu, orc, layer_spec):
    """Each sweep layer at batch 16 with the plan the benchmark runs (autotuned, then launched)."""
    ci, co, H, s = layer_spec
    x, w, bn = synthetic.dense_layer(ci, co, H, N=16, k=3)
    layer = ConvBnAct(w, bn, s, 1, cb.ACT_SILU)
    OH, OW = layer.out_hw(H, H)
    xd = to_dev(x)
    y = torch.empty(16, OH, OW, co, device=gpu)
    layer.autotune(xd, y)
    y.fill_(float("nan"))
    layer(xd, y)
    sync_check()
    ref = orc.conv_bn_act(x, w, bn, stride=s, pad=1, act=orc.ACT_SILU)
    assert rel_err(y.cpu().numpy(), ref) <= _tol(ci, co, 3, s)


@pytest.mark.parametrize("batch", [32, 1])
def test_yolo_chain_full_size_end_to_end(gpu, orc, batch):
    """The chain at 640 x 640 with the benchmark's tuned plans: final output vs the oracle chain."""
    stages = synthetic.yolo_params()
    x = synthetic.yolo_input(batch)
    chain = YoloChain(stages, batch)
    xd = to_dev(x)
    chain.forward(xd, tune=True)
    for B in chain.bufs:
        B["out"].fill_(float("nan"))
    out = chain.forward(xd)
    sync_check()
    h = x
    for st in stages:
        h = orc.yolo_stage(h, st).astype(np.float32)
    assert rel_err(out.cpu().numpy(), h) <= TOL_TF32


def test_yolo_chain_batch32_every_layer(gpu, orc):
    """Batch 32, 640 x 640: each layer (the 16- and 32-channel stage bodies, one kernel each, as one
    unit), whole output, against the oracle fed the GPU's own input (per-layer tolerance class; the
    16-channel body computes in fp32 on the CUDA cores: the fp32 bar; the 32-channel one on the
    tensor cores: the TF32 bar)."""
    stages = synthetic.yolo_params()
    x = synthetic.yolo_input(32)
    chain = YoloChain(stages, 32)
    xd = to_dev(x)
    chain.forward(xd, tune=True)
    chain.forward(xd)
    sync_check()
    h = x
    assert chain.fused[0] and chain.fused[1]
    for i, (st, B) in enumerate(zip(stages, chain.bufs)):
        half = B["half"]
        x1 = B["x1"].cpu().numpy()
        cat = B["cat"].cpu().numpy()
        out = B["out"].cpu().numpy()
        a = np.ascontiguousarray(cat[..., :half])
        checks = [("down", h, st["down_w"], st["down_bn"], 2, 1, x1, None)]
        if chain.fused[i]:
            err = rel_err(out, oracle_stage_body(orc, x1, st))
            assert err <= stage_body_tol(out.shape[-1]), f"s{i}.body: {err:.3g}"
        else:
            checks += [
                ("cv1", x1, st["cv1_w"], st["cv1_bn"], 1, 0, a, None),
                ("cv2", a, st["cv2_w"], st["cv2_bn"], 1, 1, np.ascontiguousarray(cat[..., half:]), None),
                ("cv3", cat, st["cv3_w"], st["cv3_bn"], 1, 0, out, x1),
            ]
        for name, inp, w, bn, s, p, got, res in checks:
            ref = orc.conv_bn_act(inp, w, bn, stride=s, pad=p, act=orc.ACT_SILU, residual=res,
                                  res_mode=orc.RES_POST_ACT if res is not None else orc.RES_NONE)
            err = rel_err(got, ref)
            assert err <= _tol(inp.shape[-1], w.shape[0], w.shape[2], s), f"s{i}.{name}: {err:.3g}"
        h = out


def test_preprocess_stem_full_batch32(gpu, orc):
    """32 frames 1280x720 -> 640x480 -> stem: the fused kernel against the oracle's preprocess and
    convolution; the two-kernel path's planar image bit for bit against the fp64 definition."""
    frames = synthetic.preprocess_frames(N=32)
    w, bn = synthetic.stem_params()
    net = PreprocessStem(w, bn, 32)
    fd = to_dev(frames)
    fused = net.forward(fd).cpu().numpy()
    net.forward(fd, fused=False)
    sync_check()
    planar = orc.preprocess_u8(frames, 480, 640, orc.PREC_F64)
    np.testing.assert_array_equal(net.planar.cpu().numpy(), planar)
    ref = orc.conv_bn_act(planar, w, bn, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
    assert rel_err(fused, ref) <= TOL_FP32
    assert rel_err(net.out.cpu().numpy(), ref) <= TOL_FP32


# Source -> destination extents whose scale S/D is not a dyadic rational (weights not exact in
# binary), down- and upscaling; the last ones leave exact integer sample positions (13 -> 7 at
# d = 3, 7 -> 13 at several d).
NON_DYADIC = [(100, 37), (37, 100), (13, 7), (7, 13), (720, 481), (1280, 641), (3, 7), (1000, 333)]


def _exact_coords(S, D):
    """(i0, i1, frac, exact f is an integer) per destination index, in rational arithmetic."""
    out = []
    for d in range(D):
        f = (Fraction(2 * d + 1, 2)) * Fraction(S, D) - Fraction(1, 2)
        if f < 0:
            f = Fraction(0)
        k = f.numerator // f.denominator
        t = f - k
        if k >= S - 1:
            k, t = S - 1, Fraction(0)
        out.append((k, min(k + 1, S - 1), t, t == 0))
    return out


@pytest.mark.parametrize("S,D", NON_DYADIC, ids=lambda v: str(v))
def test_preprocess_sample_coords_exact(gpu, S, D):
    """The GPU's sample indices equal the exact-rational ones; its weights are those fractions to
    within fp32 rounding of f.  Where the exact f is an integer, fp32 may land just below it: then
    (i0, frac) = (k - 1, ~1) samples the same point, which is the only other valid answer."""
    i0, i1, a = cb.debug_sample_coords(S, D)
    eps = 4 * np.finfo(np.float32).eps * (S + 1)
    for d, (k, k1, t, on_int) in enumerate(_exact_coords(S, D)):
        if i0[d] == k:
            assert i1[d] == k1, d
            assert abs(float(a[d]) - float(t)) <= eps, (d, a[d], t)
        else:
            assert on_int and i0[d] == k - 1 and 1 - float(a[d]) <= eps, (d, i0[d], k, a[d])


@pytest.mark.parametrize("S,D", [(100, 37), (37, 100), (13, 7), (7, 13), (720, 481), (1280, 641)],
                         ids=lambda v: str(v))
def test_preprocess_non_dyadic_vs_fp64_definition(gpu, orc, S, D):
    """Frames resized S x S -> D x D: every u8 code equals the fp64 definition's, except where the
    definition's value lies closer to a rounding boundary (a half-integer) than the fp32 sample
    weights can move it; there the code differs by at most one.

    The GPU evaluates f = (d + 0.5) * (S / D) - 0.5 in fp32, so its weights differ from the fp64
    definition's by |da| (read back per axis with cb_debug_sample_coords; the indices themselves
    are pinned to exact rationals above).  To first order the value then moves by
    |dax| * max(|p01 - p00|, |p11 - p10|) + |day| * |bottom - top|, plus a few fp32 roundings of
    numbers below 256: the bound used per output."""
    N = 2
    src = synthetic.frames_u8(np.random.default_rng(S * 1000 + D), (N, S, S, 3))
    dst = torch.empty(N, 3, D, D, device=gpu)
    cb.preprocess_u8(to_dev(src), dst)
    sync_check()
    got = np.rint(dst.cpu().numpy() * 255.0).astype(np.int64)          # codes k (out = k / 255)
    codes, v = orc.resize_u8(src, D, D, orc.PREC_F64, return_values=True)
    want = codes.transpose(0, 3, 1, 2).astype(np.int64)
    v = v.transpose(0, 3, 1, 2)
    gi0, _, ga = cb.debug_sample_coords(S, D)
    ei0, _, ea = orc.axis_coords(S, D, orc.PREC_F64)
    # compare weights on the same index (an exact-integer position may sit one index lower)
    da = np.where(gi0 == ei0, np.abs(ga - ea), np.abs((gi0 + ga.astype(np.float64)) - (ei0 + ea)))
    ei1 = np.minimum(ei0 + 1, S - 1)
    px = src.astype(np.float64)
    p00, p01 = px[:, ei0[:, None], ei0[None, :]], px[:, ei0[:, None], ei1[None, :]]
    p10, p11 = px[:, ei1[:, None], ei0[None, :]], px[:, ei1[:, None], ei1[None, :]]
    ax = ea[None, None, :, None]
    top, bot = (1 - ax) * p00 + ax * p01, (1 - ax) * p10 + ax * p11
    bound = (da[None, None, :, None] * np.maximum(np.abs(p01 - p00), np.abs(p11 - p10)) +
             da[None, :, None, None] * np.abs(bot - top) + 1e-3 * da.max() + 16 * 256 * np.finfo(np.float32).eps)
    bound = bound.transpose(0, 3, 1, 2)            # [N, 3, D, D] like v
    near = np.abs(v - np.floor(v) - 0.5) <= bound
    assert near.mean() < 0.1                       # the exemption stays a small set
    assert np.array_equal(got[~near], want[~near])
    assert np.all(np.abs(got[near] - want[near]) <= 1)
    # the stored value is the code divided by 255 in IEEE fp32
    table = np.arange(256, dtype=np.float32) / np.float32(255)
    assert np.array_equal(table[got], dst.cpu().numpy())
