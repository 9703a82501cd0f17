"""Layer objects and the three network chains, built from C-ABI calls.

A layer folds its BatchNorm and repacks its weights once (cb_fold_bn,
cb_repack_weights on the host), uploads them, and then every forward is one
cb_* call on preallocated device buffers, so a whole chain can be captured
in a CUDA graph (the pages' runtimes replay their inference as a graph; the
tiny MNIST layers are launch-bound without it).

  * MnistNet -- DepthwiseMNIST ("How I sped up convolutions", class listing):
    stem conv3x3 1->48 + BN + ReLU, four DepthwiseSeparableConv blocks,
    global average pool + fc 192->10.
  * YoloChain -- five stages of conv3x3 s2 -> 1x1 (C->C/2) -> 3x3 (C/2->C/2)
    -> 1x1 over the channel concat [a | b], post-activation residual; all
    conv + BN + SiLU.  The concat is fused on the producer side: the two
    branch convs write into the two channel halves of one NHWC buffer
    ("YOLO26N Inference Optimisation", improvement #6).
  * PreprocessStem -- fused u8 preprocess to planar fp32, then the stem conv
    3x3 s2 3->16 + BN + SiLU reading the planar tensor directly.
"""
from __future__ import annotations

import torch

from . import binding as cb
from .synthetic import MNIST_BLOCKS
from .workloads import out_size


def _dev(a, device):
    return torch.from_numpy(a).to(device)


class ConvBnAct:
    """One fused layer with folded BN and repacked weights on the device.

    tc_weights: prepare the dense weights for the tensor-core path -- rounded
    to the nearest TF32 value (cb_round_weights_tf32) for fp32 activations,
    converted to bf16 (cb_convert_weights_bf16) for bf16 ones; None asks the
    library (cb_layer_uses_tensor_cores) under the current kernel policy.
    dtype: the activations' storage type (torch.float32 or torch.bfloat16).
    """

    def __init__(self, w_oihw, bn, stride, pad, act, groups=1, device="cuda", eps=1e-5, tc_weights=None,
                 dtype=torch.float32):
        scale, bias = cb.fold_bn(*bn, eps=eps)
        cin = w_oihw.shape[1] * groups
        if tc_weights is None:
            tc_weights = cb.layer_uses_tensor_cores(cin, w_oihw.shape[0], w_oihw.shape[2], stride, groups)
        w = cb.repack_weights(w_oihw, groups)
        self.tc_weights = bool(tc_weights)
        self.dtype = dtype
        # host copies of the fp32 parameters as given, before any TF32 rounding or bf16 conversion
        # (calls that take their parameters from the host: cb_stage_body)
        self.w_host, self.scale_host, self.bias_host = w, scale, bias
        if tc_weights and dtype == torch.bfloat16:
            self.w = cb.convert_weights_bf16(w).to(device).contiguous()
        else:
            if tc_weights:
                w = cb.round_weights_tf32(w)
            self.w = _dev(w, device).contiguous()
        self.scale = _dev(scale, device)
        self.bias = _dev(bias, device)
        self.cout, cin_g, self.k, _ = w_oihw.shape
        self.cin = cin_g * groups
        self.stride, self.pad, self.act, self.groups = stride, pad, act, groups

    def out_hw(self, h, w):
        return out_size(h, self.k, self.stride, self.pad), out_size(w, self.k, self.stride, self.pad)

    def __call__(self, x, y, residual=None, res_mode=cb.RES_NONE, stream=None, x_layout=cb.LAYOUT_NHWC):
        return cb.conv_bn_act(x, self.w, self.scale, self.bias, self.k, self.stride, self.pad, self.groups, self.act,
                              y, residual=residual, res_mode=res_mode, stream=stream, x_layout=x_layout)

    def autotune(self, x, y, residual=None, res_mode=cb.RES_NONE, stream=None, x_layout=cb.LAYOUT_NHWC):
        """Measure this layer's tile plans on these buffers (cb_autotune_conv); later calls with the
        same shapes run the fastest.  y holds the result."""
        return cb.autotune_conv(x, self.w, self.scale, self.bias, self.k, self.stride, self.pad, self.groups,
                                self.act, y, residual=residual, res_mode=res_mode, stream=stream, x_layout=x_layout)


class DwBlock:
    """DepthwiseSeparableConv on device, run through cb_dw_separable_block."""

    def __init__(self, p, cin, cout, stride, device="cuda"):
        self.cin, self.cout, self.stride = cin, cout, stride
        dws, dwb = cb.fold_bn(*p["bn1"])
        pws, pwb = cb.fold_bn(*p["bn2"])
        pw_tc = cb.layer_uses_tensor_cores(cin, cout, 1, 1)
        skip_tc = cb.layer_uses_tensor_cores(cin, cout, 1, stride)
        dense = cb.round_weights_tf32 if pw_tc else (lambda a: a)
        dense_skip = cb.round_weights_tf32 if skip_tc else (lambda a: a)
        self.params = {
            "dw_w": _dev(cb.repack_weights(p["dw_w"], groups=cin), device),
            "dw_scale": _dev(dws, device), "dw_bias": _dev(dwb, device),
            "pw_w": _dev(dense(cb.repack_weights(p["pw_w"])), device),
            "pw_scale": _dev(pws, device), "pw_bias": _dev(pwb, device),
        }
        if "skip_w" in p:
            sks, skb = cb.fold_bn(*p["skip_bn"])
            self.params.update({"skip_w": _dev(dense_skip(cb.repack_weights(p["skip_w"])), device),
                                "skip_scale": _dev(sks, device), "skip_bias": _dev(skb, device)})

    def __call__(self, x, y, workspace, stream=None):
        return cb.dw_separable_block(x, self.params, self.stride, y, workspace, stream=stream)


class MnistNet:
    def __init__(self, params, batch, device="cuda"):
        self.batch = batch
        self.stem = ConvBnAct(params["stem_w"], params["stem_bn"], 1, 1, cb.ACT_RELU, device=device)
        self.blocks = []
        acts = [torch.empty(batch, 28, 28, 48, device=device)]
        H = 28
        ws = 0
        for blk, (cin, cout, s) in zip(params["blocks"], MNIST_BLOCKS):
            self.blocks.append(DwBlock(blk, cin, cout, s, device))
            ws = max(ws, cb.dw_separable_block_workspace(acts[-1], cout, s))
            H = out_size(H, 3, s, 1)
            acts.append(torch.empty(batch, H, H, cout, device=device))
        self.acts = acts
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=device)
        self.fc_w = _dev(params["fc_w"], device)
        self.fc_b = _dev(params["fc_b"], device)
        self.logits = torch.empty(batch, 10, device=device)

    def forward(self, x, stream=None):
        self.stem(x, self.acts[0], stream=stream)
        for i, blk in enumerate(self.blocks):
            blk(self.acts[i], self.acts[i + 1], self.workspace, stream=stream)
        cb.avgpool_linear(self.acts[-1], self.fc_w, self.fc_b, self.logits, stream=stream)
        return self.logits

    launches_per_forward = 1 + 2 + 3 + 2 + 3 + 2 + 1  # stem, blocks (dw, [skip], pw), pool+fc


class YoloChain:
    """dtype: the activations' storage type (torch.float32, or torch.bfloat16: every layer then
    reads and writes bf16, the tensor-core layers multiply bf16 weights).  fuse_body: a stage with
    16 or 32 channels runs its body (cv1, cv2, cv3 with the concat and the residual) as one kernel
    (cb_stage_body), so that a and b never reach memory; self.fused[i] says which stages do."""

    def __init__(self, stages, batch, size=640, device="cuda", dtype=torch.float32, fuse_body=True):
        self.batch = batch
        self.dtype = dtype
        self.layers = []
        self.bufs = []
        self.fused = []
        H = size
        for st in stages:
            c = st["down_w"].shape[0]
            h = c // 2
            OH = out_size(H, 3, 2, 1)
            kw = dict(device=device, dtype=dtype)
            L = {
                "down": ConvBnAct(st["down_w"], st["down_bn"], 2, 1, cb.ACT_SILU, **kw),
                "cv1": ConvBnAct(st["cv1_w"], st["cv1_bn"], 1, 0, cb.ACT_SILU, **kw),
                "cv2": ConvBnAct(st["cv2_w"], st["cv2_bn"], 1, 1, cb.ACT_SILU, **kw),
                "cv3": ConvBnAct(st["cv3_w"], st["cv3_bn"], 1, 0, cb.ACT_SILU, **kw),
            }
            B = {"x1": torch.empty(batch, OH, OH, c, device=device, dtype=dtype),
                 "cat": torch.empty(batch, OH, OH, c, device=device, dtype=dtype),
                 "out": torch.empty(batch, OH, OH, c, device=device, dtype=dtype), "half": h}
            self.layers.append(L)
            self.bufs.append(B)
            self.fused.append(fuse_body and c in (16, 32))
            H = OH

    def body(self, i, stream=None, tune=False):
        """Stage i after its stride-2 conv: x1 -> out (one kernel for a fused stage)."""
        L, B = self.layers[i], self.bufs[i]
        if self.fused[i]:
            cb.stage_body(B["x1"], (L["cv1"], L["cv2"], L["cv3"]), L["cv1"].act, B["out"], stream=stream)
            return
        half = B["half"]
        a, b = B["cat"][..., :half], B["cat"][..., half:]
        run = {k: (v.autotune if tune else v) for k, v in L.items()}
        run["cv1"](B["x1"], a, stream=stream)
        run["cv2"](a, b, stream=stream)
        run["cv3"](B["cat"], B["out"], residual=B["x1"], res_mode=cb.RES_POST_ACT, stream=stream)

    def forward(self, x, stream=None, tune=False):
        """The chain on x; tune=True measures each layer's tile plans on the way (cb_autotune_conv),
        synchronising after every layer, so that later forwards run the fastest."""
        h = x
        for i, (L, B) in enumerate(zip(self.layers, self.bufs)):
            (L["down"].autotune if tune else L["down"])(h, B["x1"], stream=stream)
            self.body(i, stream=stream, tune=tune)
            h = B["out"]
        return h

    @property
    def launches_per_forward(self):
        return sum(2 if f else 4 for f in self.fused)


class PreprocessStem:
    def __init__(self, stem_w, stem_bn, batch, src_hw=(720, 1280), dst_hw=(480, 640), device="cuda"):
        self.batch = batch
        self.src_hw, self.dst_hw = src_hw, dst_hw
        self.stem = ConvBnAct(stem_w, stem_bn, 2, 1, cb.ACT_SILU, device=device)
        Hd, Wd = dst_hw
        self.planar = torch.empty(batch, 3, Hd, Wd, device=device)
        OH, OW = self.stem.out_hw(Hd, Wd)
        self.out = torch.empty(batch, OH, OW, 16, device=device)
        self.tmp_u8 = None
        self.tmp_f32 = None

    def forward(self, frames, stream=None, three_pass=False, fused=True):
        """frames -> stem output.  fused: one kernel (cb_preprocess_stem_u8), the planar image never
        leaves shared memory; else the preprocess writes self.planar (in one pass, or in three with
        three_pass) and the stem reads it."""
        if fused and not three_pass:
            cb.preprocess_stem_u8(frames, self.dst_hw, self.stem.w, self.stem.scale, self.stem.bias, self.stem.act,
                                  self.out, stream=stream)
            return self.out
        if three_pass:
            if self.tmp_u8 is None:
                Hd, Wd = self.dst_hw
                self.tmp_u8 = torch.empty(self.batch, Hd, Wd, 3, dtype=torch.uint8, device=frames.device)
                self.tmp_f32 = torch.empty(self.batch, Hd, Wd, 3, device=frames.device)
            cb.preprocess_u8_three_pass(frames, self.tmp_u8, self.tmp_f32, self.planar, stream=stream)
        else:
            cb.preprocess_u8(frames, self.planar, stream=stream)
        self.stem(self.planar, self.out, stream=stream, x_layout=cb.LAYOUT_NCHW)
        return self.out
