"""GPU parity: u8 frame preprocess, fused and three-pass, vs the oracle.

The u8 code is an integer decided by floating point, so both sides decide in
the kernel's precision (IEEE fp32, each operation rounded, no fused
multiply-add): the oracle's PREC_F32 mode.  Bar: bit-exact.
"""
import numpy as np
import pytest
import torch

from conv_bn_activation_gb300 import binding as cb, synthetic
from gpu_util import sync_check, to_dev

pytestmark = pytest.mark.gpu

SIZES = [(720, 1280, 480, 640), (13, 17, 7, 9), (100, 37, 41, 100), (64, 64, 64, 64), (9, 5, 31, 33),
         (480, 640, 480, 640), (1, 1, 3, 4), (5, 1000, 3, 333),
         # exact 2:1 widths (the pair-sum path) with odd, equal, upscaled and downscaled heights
         (15, 64, 7, 32), (8, 40, 20, 20), (31, 80, 31, 40), (9, 16, 2, 8), (2, 24, 5, 12)]


@pytest.mark.parametrize("size", SIZES, ids=lambda s: "%dx%d-%dx%d" % s)
def test_preprocess_bit_exact(gpu, orc, size):
    Hs, Ws, Hd, Wd = size
    N = 2
    src = synthetic.frames_u8(np.random.default_rng(Hs * Ws), (N, Hs, Ws, 3))
    dst = torch.empty(N, 3, Hd, Wd, device=gpu)
    cb.preprocess_u8(to_dev(src), dst)
    sync_check()
    ref = orc.preprocess_u8(src, Hd, Wd, orc.PREC_F32)
    np.testing.assert_array_equal(dst.cpu().numpy(), ref)
    # three-pass path: same bits
    tmp_u8 = torch.empty(N, Hd, Wd, 3, dtype=torch.uint8, device=gpu)
    tmp_f32 = torch.empty(N, Hd, Wd, 3, device=gpu)
    dst3 = torch.empty_like(dst)
    cb.preprocess_u8_three_pass(to_dev(src), tmp_u8, tmp_f32, dst3)
    sync_check()
    np.testing.assert_array_equal(dst3.cpu().numpy(), ref)
    np.testing.assert_array_equal(tmp_u8.cpu().numpy(), orc.resize_u8(src, Hd, Wd, orc.PREC_F32))


def test_preprocess_padded_pitch(gpu, orc):
    """Source rows padded past 3*W bytes (pitch 3*W + 37): the padding is never read into the result."""
    N, Hs, Ws, Hd, Wd = 2, 30, 50, 20, 24
    src = synthetic.frames_u8(np.random.default_rng(9), (N, Hs, Ws, 3))
    pitch = Ws * 3 + 37
    buf = torch.full((N, Hs, pitch), 255, dtype=torch.uint8)
    buf[:, :, :Ws * 3] = torch.from_numpy(src.reshape(N, Hs, Ws * 3))
    buf = buf.to(gpu)
    view = torch.as_strided(buf, (N, Hs, Ws, 3), (Hs * pitch, pitch, 3, 1))
    dst = torch.empty(N, 3, Hd, Wd, device=gpu)
    cb.preprocess_u8(view, dst)
    sync_check()
    np.testing.assert_array_equal(dst.cpu().numpy(), orc.preprocess_u8(src, Hd, Wd, orc.PREC_F32))


def test_preprocess_workload_frames(gpu, orc):
    """Four frames of the 1280x720 -> 640x480 workload: fp32 decisions equal fp64 ones at this ratio,
    so the GPU output equals the fp64 definition bit for bit."""
    src = synthetic.preprocess_frames(N=4)
    dst = torch.empty(4, 3, 480, 640, device=gpu)
    cb.preprocess_u8(to_dev(src), dst)
    sync_check()
    np.testing.assert_array_equal(dst.cpu().numpy(), orc.preprocess_u8(src, 480, 640, orc.PREC_F64))


def test_preprocess_full_batch_properties(gpu):
    """Batch 32 (the bench launch): every output is k/255 for an integer k in [0, 255]."""
    src = synthetic.preprocess_frames(N=32)
    dst = torch.empty(32, 3, 480, 640, device=gpu)
    cb.preprocess_u8(to_dev(src), dst)
    sync_check()
    k = torch.round(dst * 255)
    assert bool(((k >= 0) & (k <= 255)).all())
    table = torch.from_numpy(np.arange(256, dtype=np.float32) / np.float32(255)).to(gpu)  # IEEE u / 255
    assert bool((table[k.long()] == dst).all())
