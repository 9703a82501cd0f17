"""Pins for the oracle's BatchNorm, activations and residual placement (CPU only).

BN is the unfolded inference form gamma*(z-mean)/sqrt(var+eps)+beta ("How I
sped up convolutions", Metal kernel step 4).  SiLU is z*sigmoid(z) (the pages
name it without a definition).  Residual placement: pre-activation
relu(bn + identity) in DepthwiseSeparableConv.forward; post-activation for
the YOLO-style chain.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch


def test_bn_closed_forms(orc):
    C = 4
    gamma = np.array([0.5, 1.0, 1.5, 2.0], np.float32)
    beta = np.array([0.1, -0.2, 0.0, 0.3], np.float32)
    mean = np.array([0.25, -0.5, 1.0, 0.0], np.float32)
    var = np.array([1.0, 0.75, 4.0, 0.5], np.float32)
    eps = 1e-5
    sd = np.sqrt(var.astype(np.float64) + eps)
    # z = mean -> beta ; z = mean + sqrt(var+eps) -> gamma + beta
    z = np.stack([mean.astype(np.float64), mean + sd])
    out = orc.batchnorm(z, gamma, beta, mean, var, eps)
    np.testing.assert_allclose(out[0], beta, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[1], gamma.astype(np.float64) + beta, rtol=1e-15, atol=1e-15)


def test_bn_identity_parameters(orc):
    """gamma=1, beta=0, mean=0, var=1-eps is the identity."""
    eps = 0.25  # exactly representable, so var + eps == 1 exactly
    C = 3
    z = np.random.default_rng(0).standard_normal((10, C))
    out = orc.batchnorm(z, np.ones(C), np.zeros(C), np.zeros(C), np.full(C, 0.75), eps)
    np.testing.assert_array_equal(out, z)


def test_bn_matches_torch_batchnorm_eval(orc):
    g = np.random.default_rng(1)
    C = 7
    z = g.standard_normal((2, 5, 6, C))
    gamma, var = (g.uniform(0.5, 1.5, C).astype(np.float32) for _ in range(2))
    beta, mean = ((g.standard_normal(C) * 0.1).astype(np.float32) for _ in range(2))
    bn = torch.nn.BatchNorm2d(C, eps=1e-5).double().eval()
    with torch.no_grad():
        bn.weight.copy_(torch.from_numpy(gamma.astype(np.float64)))
        bn.bias.copy_(torch.from_numpy(beta.astype(np.float64)))
        bn.running_mean.copy_(torch.from_numpy(mean.astype(np.float64)))
        bn.running_var.copy_(torch.from_numpy(var.astype(np.float64)))
        ref = bn(torch.from_numpy(z).permute(0, 3, 1, 2)).permute(0, 2, 3, 1).numpy()
    np.testing.assert_allclose(orc.batchnorm(z, gamma, beta, mean, var), ref, rtol=1e-13, atol=1e-13)


def test_relu_closed_forms(orc):
    v = np.array([-3.0, -0.0, 0.0, 1e-300, 2.5, 1e30])
    np.testing.assert_array_equal(orc.activation(v, orc.ACT_RELU), [0, 0, 0, 1e-300, 2.5, 1e30])
    np.testing.assert_array_equal(orc.activation(v, orc.ACT_NONE), v)


def test_silu_closed_forms(orc):
    ln3 = math.log(3.0)
    v = np.array([0.0, ln3, -ln3, 800.0, -800.0])
    out = orc.activation(v, orc.ACT_SILU)
    # sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4
    np.testing.assert_allclose(out[:3], [0.0, 0.75 * ln3, -0.25 * ln3], rtol=1e-15, atol=1e-16)
    assert out[3] == 800.0 and out[4] == 0.0


def test_silu_odd_identity_and_library(orc):
    v = np.random.default_rng(2).standard_normal(1000) * 8
    s = orc.activation(v, orc.ACT_SILU)
    sm = orc.activation(-v, orc.ACT_SILU)
    np.testing.assert_allclose(s - sm, v, rtol=1e-13, atol=1e-13)   # silu(x) - silu(-x) = x
    np.testing.assert_allclose(s, v * scipy.special.expit(v), rtol=1e-14, atol=1e-300)


def _params(g, C):
    return (g.uniform(0.5, 1.5, C).astype(np.float32), (g.standard_normal(C) * 0.1).astype(np.float32),
            (g.standard_normal(C) * 0.1).astype(np.float32), g.uniform(0.5, 1.5, C).astype(np.float32))


@pytest.mark.parametrize("act", [0, 1, 2])
def test_residual_placement(orc, act):
    g = np.random.default_rng(3 + act)
    x = g.standard_normal((1, 6, 5, 4)).astype(np.float32)
    w = g.standard_normal((4, 4, 3, 3)).astype(np.float32)
    bn = _params(g, 4)
    r = g.standard_normal((1, 6, 5, 4)).astype(np.float32)
    base = orc.batchnorm(orc.conv2d(x, w, pad=1), *bn)
    pre = orc.conv_bn_act(x, w, bn, pad=1, act=act, residual=r, res_mode=orc.RES_PRE_ACT)
    post = orc.conv_bn_act(x, w, bn, pad=1, act=act, residual=r, res_mode=orc.RES_POST_ACT)
    none = orc.conv_bn_act(x, w, bn, pad=1, act=act)
    np.testing.assert_array_equal(none, orc.activation(base, act))
    np.testing.assert_array_equal(pre, orc.activation(base + r, act))
    np.testing.assert_array_equal(post, orc.activation(base, act) + r)
    if act == orc.ACT_NONE:
        np.testing.assert_array_equal(pre, post)


def test_zero_weights_give_activated_bias(orc):
    """w = 0 => y = act(beta - gamma*mean/sqrt(var+eps) [+ r])."""
    g = np.random.default_rng(9)
    C = 5
    bn = _params(g, C)
    x = g.standard_normal((2, 4, 4, 3)).astype(np.float32)
    w = np.zeros((C, 3, 3, 3), np.float32)
    r = g.standard_normal((2, 2, 2, C)).astype(np.float32)
    gamma, beta, mean, var = (b.astype(np.float64) for b in bn)
    shift = beta - gamma * mean / np.sqrt(var + 1e-5)
    y = orc.conv_bn_act(x, w, bn, stride=2, pad=1, act=orc.ACT_SILU, residual=r, res_mode=orc.RES_PRE_ACT)
    v = shift + r
    np.testing.assert_allclose(y, v / (1 + np.exp(-v)), rtol=1e-14, atol=1e-15)
