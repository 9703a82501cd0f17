"""GPU parity of the three network chains against the oracle chains.

Tolerance bookkeeping: a chain containing tensor-core (TF32) layers is held
to 5e-3 relative to max end to end; per-layer checks feed the oracle the
GPU's own input.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from conv_bn_activation_gb300.nets import MnistNet, PreprocessStem, YoloChain
from gpu_util import TOL_FP32, TOL_TF32, oracle_stage_body, rel_err, stage_body_tol, sync_check, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("batch", [64, 3])
def test_mnist_forward(gpu, orc, batch):
    params = synthetic.mnist_params()
    x = synthetic.mnist_input(batch)
    net = MnistNet(params, batch)
    logits = net.forward(to_dev(x)).clone()
    sync_check()
    ref = orc.mnist_model(x, params)
    assert rel_err(logits.cpu().numpy(), ref) <= TOL_TF32


def test_mnist_graph_replay_matches_eager(gpu):
    params = synthetic.mnist_params()
    x = to_dev(synthetic.mnist_input(64))
    net = MnistNet(params, 64)
    eager = net.forward(x).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        net.forward(x)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        net.forward(x)
    net.logits.zero_()
    g.replay()
    sync_check()
    assert torch.equal(net.logits, eager)


@pytest.mark.parametrize("fuse_body", [True, False], ids=["fused_body", "layers"])
def test_yolo_chain_small(gpu, orc, fuse_body):
    """The chain end to end at 96 x 96, with the 16- and 32-channel stage bodies as one kernel each
    or as their three layers."""
    stages = synthetic.yolo_params()
    x = synthetic.yolo_input(2, size=96)
    chain = YoloChain(stages, 2, size=96, fuse_body=fuse_body)
    assert chain.fused[:2] == [fuse_body] * 2 and not any(chain.fused[2:])
    assert chain.launches_per_forward == (16 if fuse_body else 20)
    out = chain.forward(to_dev(x))
    sync_check()
    h = x
    for st in stages:
        h = orc.yolo_stage(h, st).astype(np.float32)
    assert rel_err(out.cpu().numpy(), h) <= TOL_TF32


def test_yolo_chain_full_size_per_layer(gpu, orc):
    """640x640, batch 1: each layer's GPU output vs the oracle fed the GPU's own input (sampled)."""
    stages = synthetic.yolo_params()
    x = synthetic.yolo_input(1)
    chain = YoloChain(stages, 1)
    chain.forward(to_dev(x))
    sync_check()
    rng = np.random.default_rng(0)
    h = x
    for i, (st, B) in enumerate(zip(stages, chain.bufs)):
        half = B["half"]
        x1 = B["x1"].cpu().numpy()
        cat = B["cat"].cpu().numpy()
        out = B["out"].cpu().numpy()
        checks = [(h, st["down_w"], st["down_bn"], 2, 1, x1, None)]
        if chain.fused[i]:  # the body as one unit (a and b never reach memory)
            assert rel_err(out, oracle_stage_body(orc, x1, st)) <= stage_body_tol(out.shape[-1])
        else:
            checks += [
                (x1, st["cv1_w"], st["cv1_bn"], 1, 0, cat[..., :half], None),
                (np.ascontiguousarray(cat[..., :half]), st["cv2_w"], st["cv2_bn"], 1, 1, cat[..., half:], None),
                (cat, st["cv3_w"], st["cv3_bn"], 1, 0, out, x1),
            ]
        for inp, w, bn, s, p, got, res in checks:
            got = np.ascontiguousarray(got)
            idx = rng.choice(got.size, min(got.size, 3000), replace=False)
            ref = orc.conv_bn_act_points(inp, w, bn, idx, stride=s, pad=p, act=orc.ACT_SILU, residual=res,
                                         res_mode=orc.RES_POST_ACT if res is not None else orc.RES_NONE)
            tc = cb.layer_uses_tensor_cores(inp.shape[-1], w.shape[0], w.shape[2], s)
            tol = TOL_TF32 if tc else TOL_FP32
            assert rel_err(got.reshape(-1)[idx], ref) <= tol
        h = out


@pytest.mark.parametrize("mode", ["fused", "two_kernel", "three_pass"])
def test_preprocess_stem(gpu, orc, mode):
    frames = synthetic.preprocess_frames(N=2)
    w, bn = synthetic.stem_params()
    net = PreprocessStem(w, bn, 2)
    out = net.forward(to_dev(frames), three_pass=mode == "three_pass", fused=mode == "fused")
    sync_check()
    planar = orc.preprocess_u8(frames, 480, 640, orc.PREC_F32)
    if mode != "fused":
        np.testing.assert_array_equal(net.planar.cpu().numpy(), planar)
    ref = orc.conv_bn_act(planar, w, bn, stride=2, pad=1, act=orc.ACT_SILU, layout=orc.NCHW)
    assert rel_err(out.cpu().numpy(), ref) <= TOL_FP32
