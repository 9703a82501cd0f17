"""Pins for the oracle's block and model compositions (CPU only).

DepthwiseMNIST / DepthwiseSeparableConv structure: "How I sped up
convolutions", class listings.  YOLO-style stage: the five-stage chain of
conv3x3 s2 -> 1x1 (C->C/2) -> 3x3 (C/2->C/2) -> 1x1 over the concat [a|b]
with a post-activation residual (the plain reading of "followed by ... plus
residual add").  The torch references here are written with torch.nn.functional
in float64 as independent library formulations.
"""
import json
import os

import numpy as np
import torch
import torch.nn.functional as F

from conv_bn_activation_gb300 import synthetic, workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def _bn(z, bn, eps=1e-5):
    g, b, m, v = (_t(p) for p in bn)
    return F.batch_norm(z, m, v, g, b, training=False, eps=eps)


def _torch_block(x, p, stride):
    cin = x.shape[1]
    cout = p["pw_w"].shape[0]
    t = F.relu(_bn(F.conv2d(x, _t(p["dw_w"]), stride=stride, padding=1, groups=cin), p["bn1"]))
    u = _bn(F.conv2d(t, _t(p["pw_w"])), p["bn2"])
    ident = _bn(F.conv2d(x, _t(p["skip_w"]), stride=stride), p["skip_bn"]) if (stride != 1 or cin != cout) else x
    return F.relu(u + ident)


def _torch_mnist(x_nhwc, params):
    x = _t(x_nhwc).permute(0, 3, 1, 2)
    h = F.relu(_bn(F.conv2d(x, _t(params["stem_w"]), padding=1), params["stem_bn"]))
    for blk, (_, _, s) in zip(params["blocks"], synthetic.MNIST_BLOCKS):
        h = _torch_block(h, blk, s)
    pooled = h.mean(dim=(2, 3))
    return pooled @ _t(params["fc_w"]).T + _t(params["fc_b"])


def test_mnist_forward_matches_torch(orc):
    params = synthetic.mnist_params()
    x = synthetic.mnist_input(batch=3)
    got = orc.mnist_model(x, params)
    ref = _torch_mnist(x, params).numpy()
    assert got.shape == (3, 10)
    # the oracle stores inter-layer activations in fp32; the torch reference keeps fp64
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * np.abs(ref).max())


def test_mnist_param_count():
    params = synthetic.mnist_params()
    import oracle
    n = oracle.mnist_param_count(params)
    # closed form: stem 48*9 + BN 2*48; blocks dw C*9 + 2C, pw Cout*Cin + 2Cout, skip Cout*Cin + 2Cout
    want = 48 * 9 + 96
    for cin, cout, s in synthetic.MNIST_BLOCKS:
        want += cin * 9 + 2 * cin + cout * cin + 2 * cout
        if s != 1 or cin != cout:
            want += cout * cin + 2 * cout
    want += 192 * 10 + 10
    assert n == want == 101_098
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["mnist_params_approx"]
    assert abs(n - g["value"]) / g["value"] < g["tolerance_rel"]


def test_mnist_flops_near_page_figure():
    f = workloads.total(workloads.mnist_layers(N=1)).flops
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["mnist_flops_per_pass_approx"]
    assert f == 15_903_360
    assert abs(f - g["value"]) / g["value"] < g["tolerance_rel"]


def test_depthwise_intensity_range():
    """Our depthwise byte model gives 0.90 (stride 2) to 2.25 (stride 1) FLOP/B; the page quotes 0.87-2.2."""
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["depthwise_intensity_range"]
    lo, hi = g["value"]
    ai = [w.intensity for name, w in workloads.mnist_layers(N=64) if name.endswith(".dw")]
    assert abs(min(ai) - lo) < g["tolerance_abs"] and abs(max(ai) - hi) < g["tolerance_abs"]
    dw = workloads.depthwise_workload()
    assert abs(dw["s1"].intensity - 2.25) < 0.001 and abs(dw["s2"].intensity - 0.90) < 0.001
    assert dw["s1"].bytes - 2 * 64 * 56 * 56 * 384 * 4 == 384 * 9 * 4 + 2 * 384 * 4


def test_bf16_storage_byte_ledger():
    """bf16 storage halves the activation bytes of a layer (input, output, residual) and leaves
    the fp32 weights, scale and bias; the FLOPs do not change."""
    f32, b16 = workloads.depthwise_workload(), workloads.depthwise_workload(act_bytes=2)
    for k in ("s1", "s2"):
        params = 384 * 9 * 4 + 2 * 384 * 4
        assert b16[k].flops == f32[k].flops
        assert b16[k].bytes - params == (f32[k].bytes - params) // 2
    assert b16["s1"].bytes == 308298240  # the bench's algorithmic bytes for the bf16 stride-1 launch
    pw32 = workloads.conv_layer(32, 320, 320, 16, 16, 1, 1, 0, residual=True)
    pw16 = workloads.conv_layer(32, 320, 320, 16, 16, 1, 1, 0, residual=True, act_bytes=2)
    params = 16 * 16 * 4 + 2 * 16 * 4
    assert pw16.bytes - params == (pw32.bytes - params) // 2 == 3 * 32 * 320 * 320 * 16 * 2


def _torch_stage(x, st):
    x1 = F.silu(_bn(F.conv2d(x, _t(st["down_w"]), stride=2, padding=1), st["down_bn"]))
    a = F.silu(_bn(F.conv2d(x1, _t(st["cv1_w"])), st["cv1_bn"]))
    b = F.silu(_bn(F.conv2d(a, _t(st["cv2_w"]), padding=1), st["cv2_bn"]))
    return F.silu(_bn(F.conv2d(torch.cat([a, b], 1), _t(st["cv3_w"])), st["cv3_bn"])) + x1


def test_yolo_stage_matches_torch_and_shapes(orc):
    stages = synthetic.yolo_params()
    x = synthetic.yolo_input(1, size=64)
    h = x
    widths = []
    for st in stages:
        ref = _torch_stage(_t(h).permute(0, 3, 1, 2), st).permute(0, 2, 3, 1).numpy()
        got = orc.yolo_stage(h, st)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-5 * np.abs(ref).max())
        widths.append(got.shape[2])
        h = got.astype(np.float32)
    assert widths == [32, 16, 8, 4, 2]
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["yolo_stem_output"]["value"]
    assert [name for name, _ in workloads.yolo_layers()][:4] == ["s0.down", "s0.cv1", "s0.cv2", "s0.cv3"]
    assert len(workloads.yolo_layers()) == 20
    sizes = [640 // 2 ** (i + 1) for i in range(5)]
    assert sizes == g


def test_tma_overflow_arithmetic():
    """A 16-wide tile over rows of OW=40 / 20 overshoots by 8 / 12 columns; padding rows to a
    multiple of 16 absorbs exactly that overshoot."""
    g = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["tma_overflow_columns"]
    B = g["block_ow"]
    for ow, spill in g["value"].items():
        ow = int(ow)
        assert (-ow) % B == spill
        assert ((ow + B - 1) // B) * B - ow == spill
