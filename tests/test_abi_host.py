"""Host-side checks of the C ABI (CPU only: no kernel is launched).

The library must load and export every entry point include/cb.h declares;
the host helpers (BN folding, weight repacking) are checked against the
oracle and numpy; invalid arguments are rejected before any launch.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "cb.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cb_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(cblib):
    lib = cblib.load()
    names = _declared()
    assert "cb_conv_bn_act" in names and "cb_preprocess_u8" in names and "cb_fold_bn" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(cblib.EXPORTED)
    assert cblib.version() >= 100


def test_status_strings(cblib):
    assert cblib.status_string(cblib.OK) == "CB_OK"
    assert cblib.status_string(cblib.ERR_TIMEOUT) == "CB_ERR_TIMEOUT"


def test_fold_bn_matches_unfolded_oracle(cblib, orc):
    """Folded (scale, bias) applied to z equals the oracle's unfolded BN to fp32 rounding."""
    g = np.random.default_rng(0)
    C = 37
    gamma, var = g.uniform(0.5, 1.5, C).astype(np.float32), g.uniform(0.5, 1.5, C).astype(np.float32)
    beta, mean = (g.standard_normal(C) * 0.1).astype(np.float32), (g.standard_normal(C) * 0.1).astype(np.float32)
    scale, bias = cblib.fold_bn(gamma, beta, mean, var, 1e-5)
    z = g.standard_normal((50, C)) * 3
    folded = z * scale.astype(np.float64) + bias.astype(np.float64)
    unfolded = orc.batchnorm(z, gamma, beta, mean, var, 1e-5)
    # only the fp32 storage of (scale, bias) separates them
    assert np.max(np.abs(folded - unfolded)) < 4e-7 * (np.max(np.abs(unfolded)) + 1)


def test_fold_bn_rejects_bad_args(cblib):
    lib = cblib.load()
    v = np.ones(4, np.float32)
    out = np.empty(4, np.float32)
    neg = np.full(4, -1.0, np.float32)
    assert lib.cb_fold_bn(v.ctypes.data, v.ctypes.data, v.ctypes.data, neg.ctypes.data, ctypes.c_float(1e-5), 4,
                          out.ctypes.data, out.ctypes.data) == cblib.ERR_INVALID_ARG
    assert lib.cb_fold_bn(None, v.ctypes.data, v.ctypes.data, v.ctypes.data, ctypes.c_float(1e-5), 4,
                          out.ctypes.data, out.ctypes.data) == cblib.ERR_INVALID_ARG
    assert lib.cb_fold_bn(v.ctypes.data, v.ctypes.data, v.ctypes.data, v.ctypes.data, ctypes.c_float(1e-5), 0,
                          out.ctypes.data, out.ctypes.data) == cblib.ERR_INVALID_ARG


def test_repack_is_exact_permutation(cblib):
    g = np.random.default_rng(1)
    w = g.standard_normal((6, 5, 3, 3)).astype(np.float32)
    np.testing.assert_array_equal(cblib.repack_weights(w), w.transpose(0, 2, 3, 1))
    wd = g.standard_normal((7, 1, 3, 3)).astype(np.float32)
    np.testing.assert_array_equal(cblib.repack_weights(wd, groups=7), wd[:, 0].transpose(1, 2, 0))
    w1 = g.standard_normal((4, 8, 1, 1)).astype(np.float32)
    np.testing.assert_array_equal(cblib.repack_weights(w1).reshape(4, 8), w1[:, :, 0, 0])
    with pytest.raises(cblib.CbError):
        cblib.repack_weights(g.standard_normal((8, 2, 3, 3)).astype(np.float32), groups=4)


def _view(data, n, h, w, c, layout=0):
    if layout == 0:
        return __import__("conv_bn_activation_gb300").binding.CbTensor(data, n, h, w, c, h * w * c, w * c, c, 1, 0)
    return __import__("conv_bn_activation_gb300").binding.CbTensor(data, n, h, w, c, c * h * w, w, 1, h * w, 1)


def test_conv_rejects_invalid_arguments_before_launch(cblib):
    lib = cblib.load()
    T = ctypes.byref
    base = 1 << 20  # fake, never dereferenced: validation fails first
    x = _view(base, 1, 8, 8, 16)
    y_ok = _view(base + (1 << 16), 1, 8, 8, 16)
    w = s = b = base + (1 << 18)
    call = lambda xv, yv, k=3, st=1, p=1, g=1, act=0, r=None, rm=0: lib.cb_conv_bn_act(
        T(xv), w, s, b, k, k, st, p, g, act, T(r) if r is not None else None, rm, T(yv), None)
    assert call(x, _view(base + (1 << 16), 1, 7, 8, 16)) == cblib.ERR_INVALID_ARG        # wrong OH
    assert call(x, y_ok, k=5, p=2) == cblib.ERR_UNSUPPORTED                             # 5x5
    assert call(x, y_ok, st=3) == cblib.ERR_UNSUPPORTED                                 # stride 3
    assert call(x, y_ok, g=4) == cblib.ERR_UNSUPPORTED                                  # groups 4
    assert call(x, y_ok, act=7) == cblib.ERR_INVALID_ARG                                # bad act
    assert call(x, y_ok, rm=1) == cblib.ERR_INVALID_ARG                                 # residual missing
    assert call(x, _view(base + 64, 1, 8, 8, 16)) == cblib.ERR_INVALID_ARG              # x / y overlap
    assert call(x, y_ok, r=_view(base + (1 << 16) + 4, 1, 8, 8, 16), rm=1) == cblib.ERR_INVALID_ARG  # r partly on y
    bad = _view(base, 1, 8, 8, 16)
    bad.stride_c = 2
    assert call(bad, y_ok) == cblib.ERR_INVALID_ARG                                     # NHWC needs unit c stride
    assert lib.cb_conv_bn_act(T(x), None, s, b, 3, 3, 1, 1, 1, 0, None, 0, T(y_ok), None) == cblib.ERR_INVALID_ARG
    # empty batch: valid, nothing to do, no launch
    assert call(_view(base, 0, 8, 8, 16), _view(base + (1 << 16), 0, 8, 8, 16)) == cblib.OK


def test_bf16_views_validated_before_launch(cblib):
    """bf16 storage: depthwise 3x3 and narrow 1x1 layers only, every view the same element type,
    unknown element types rejected -- all decided on the host (fake pointers, never dereferenced)."""
    lib = cblib.load()
    T = ctypes.byref
    base = 1 << 20
    w = s = b = base + (1 << 18)

    def v(data, n, h, w_, c, dtype):
        t = _view(data, n, h, w_, c)
        t.dtype = dtype
        return t
    x16 = v(base, 1, 8, 8, 16, cblib.DTYPE_BF16)
    y16 = v(base + (1 << 16), 1, 8, 8, 16, cblib.DTYPE_BF16)
    y32 = v(base + (1 << 16), 1, 8, 8, 16, cblib.DTYPE_F32)
    call = lambda xv, yv, g=1, r=None, rm=0: lib.cb_conv_bn_act(
        T(xv), w, s, b, 3, 3, 1, 1, g, 0, T(r) if r is not None else None, rm, T(yv), None)
    x12 = v(base, 1, 8, 8, 12, cblib.DTYPE_BF16)
    assert call(x12, v(base + (1 << 16), 1, 8, 8, 12, cblib.DTYPE_BF16), g=1) == cblib.ERR_UNSUPPORTED  # 3x3, 12 ch
    assert call(x16, y32, g=16) == cblib.ERR_INVALID_ARG                     # mixed element types
    assert call(x16, y16, g=16, r=v(base + (1 << 17), 1, 8, 8, 16, cblib.DTYPE_F32), rm=2) == cblib.ERR_INVALID_ARG
    assert call(v(base, 1, 8, 8, 16, 7), v(base + (1 << 16), 1, 8, 8, 16, 7), g=16) == cblib.ERR_INVALID_ARG
    assert lib.cb_conv_path(T(x16), T(y16), 3, 1, 1, 16) == cblib.PATH_DEPTHWISE
    assert lib.cb_conv_path(T(x16), T(y16), 1, 1, 0, 1) == cblib.PATH_POINTWISE   # 1x1 16 -> 16
    x4 = v(base, 1, 8, 8, 4, cblib.DTYPE_BF16)
    assert lib.cb_conv_bn_act(T(x4), w, s, b, 1, 1, 1, 0, 1, 0, None, 0, T(v(base + (1 << 16), 1, 8, 8, 16, cblib.DTYPE_BF16)),
                              None) == cblib.ERR_UNSUPPORTED                   # 1x1 bf16 needs Ci >= 8
    assert lib.cb_conv_path(T(x16), T(y16), 3, 1, 1, 1) == 0
    assert lib.cb_conv_path(T(x16), T(y32), 3, 1, 1, 16) == 0
    # empty bf16 depthwise batch: valid, nothing to launch
    assert call(v(base, 0, 8, 8, 16, cblib.DTYPE_BF16), v(base + 8 * 8 * 16 * 2, 0, 8, 8, 16, cblib.DTYPE_BF16),
                g=16) == cblib.OK
    n = ctypes.c_size_t(0)
    assert lib.cb_dw_separable_block_workspace(T(x16), 16, 1, T(n)) == cblib.ERR_UNSUPPORTED


def test_binding_dtype_codes(cblib):
    import torch
    assert cblib.dtype_code(torch.empty(1)) == cblib.DTYPE_F32
    assert cblib.dtype_code(torch.empty(1, dtype=torch.bfloat16)) == cblib.DTYPE_BF16
    with pytest.raises(TypeError):
        cblib.dtype_code(torch.empty(1, dtype=torch.float16))
    assert cblib.nhwc(torch.empty(1, 2, 3, 8, dtype=torch.bfloat16)).dtype == cblib.DTYPE_BF16


def test_block_and_preprocess_validation(cblib):
    lib = cblib.load()
    T = ctypes.byref
    base = 1 << 20
    x = _view(base, 2, 14, 14, 48)
    y = _view(base + (1 << 22), 2, 7, 7, 96)
    n = ctypes.c_size_t(0)
    assert lib.cb_dw_separable_block_workspace(T(x), 96, 2, T(n)) == cblib.OK
    rup = lambda b: (b + 255) // 256 * 256
    assert n.value == rup(2 * 7 * 7 * 48 * 4) + rup(2 * 7 * 7 * 96 * 4)
    p = base + (1 << 24)
    # too-small workspace
    assert lib.cb_dw_separable_block(T(x), p, p, p, p, p, p, p, p, p, 2, T(y), p, 16, None) == cblib.ERR_WORKSPACE
    # identity skip needs stride 1 and Cin == Cout
    assert lib.cb_dw_separable_block(T(x), p, p, p, p, p, p, None, None, None, 2, T(y), p, n.value,
                                     None) == cblib.ERR_INVALID_ARG
    # preprocess: pitch smaller than a row
    assert lib.cb_preprocess_u8(base, 1, 720, 1280, 1000, base + (1 << 24), 480, 640, None) == cblib.ERR_INVALID_ARG
    assert lib.cb_preprocess_u8(None, 1, 720, 1280, 3840, base, 480, 640, None) == cblib.ERR_INVALID_ARG


def test_stage_body_validated_before_launch(cblib):
    """cb_stage_body: NULL weights, shape, dtype and overlap errors, unsupported channel counts and
    layouts, and misaligned strides are all decided on the host (fake pointers, never read)."""
    lib = cblib.load()
    T = ctypes.byref
    base = 1 << 20
    p = base + (1 << 24)
    x = _view(base, 2, 16, 32, 16)
    y = _view(base + (1 << 22), 2, 16, 32, 16)
    call = lambda xv, yv, w=p, act=2: lib.cb_stage_body(T(xv), w, p, p, p, p, p, p, p, p, act, T(yv), None)
    assert call(x, y, w=None) == cblib.ERR_INVALID_ARG                                   # NULL weights
    assert call(x, y, act=5) == cblib.ERR_INVALID_ARG                                    # bad act
    assert call(x, _view(base + (1 << 22), 2, 16, 31, 16)) == cblib.ERR_INVALID_ARG      # shape mismatch
    assert call(x, _view(base + 64, 2, 16, 32, 16)) == cblib.ERR_INVALID_ARG             # y overlaps x1
    assert call(_view(base, 2, 16, 32, 8), _view(base + (1 << 22), 2, 16, 32, 8)) == cblib.ERR_UNSUPPORTED
    odd = _view(base, 2, 16, 32, 16)
    odd.stride_w, odd.stride_h, odd.stride_n = 18, 18 * 32, 18 * 32 * 16                  # pixels 72 bytes apart
    assert call(odd, y) == cblib.ERR_ALIGNMENT
    assert call(_view(base, 0, 16, 32, 16), _view(base + (1 << 22), 0, 16, 32, 16)) == cblib.OK  # empty batch
    # 32 channels (the tensor-core body): y strides in whole 16-byte pieces (its tensor stores)
    x32, y32 = _view(base, 2, 16, 32, 32), _view(base + (1 << 22), 2, 16, 32, 32)
    assert call(_view(base, 2, 16, 32, 24), _view(base + (1 << 22), 2, 16, 32, 24)) == cblib.ERR_UNSUPPORTED
    xb, yb = _view(base, 2, 16, 32, 32), _view(base + (1 << 22), 2, 16, 32, 32)
    xb.dtype = yb.dtype = cblib.DTYPE_BF16
    yb.stride_w, yb.stride_h, yb.stride_n = 36, 36 * 32, 36 * 32 * 16                   # bf16 y pixels 72 bytes apart
    assert call(xb, yb) == cblib.ERR_ALIGNMENT
    odd32 = _view(base + (1 << 22), 2, 16, 32, 32)
    odd32.stride_w, odd32.stride_h, odd32.stride_n = 34, 34 * 32, 34 * 32 * 16              # y pixels 136 bytes apart
    assert call(x32, odd32) == cblib.ERR_ALIGNMENT
    assert call(x32, _view(base + 64, 2, 16, 32, 32)) == cblib.ERR_INVALID_ARG            # y overlaps x1
    assert call(_view(base, 0, 16, 32, 32), _view(base + (1 << 22), 0, 16, 32, 32)) == cblib.OK  # empty batch


def test_round_weights_tf32(cblib):
    """Round to nearest TF32 (ties to even): low 13 mantissa bits clear, error <= half a TF32 ulp,
    idempotent, and the tie cases go to the even neighbour."""
    g = np.random.default_rng(2)
    w = (g.standard_normal(10000) * np.exp(g.uniform(-20, 20, 10000))).astype(np.float32)
    r = cblib.round_weights_tf32(w)
    bits = r.view(np.uint32)
    assert np.all(bits & 0x1FFF == 0)
    ulp = np.spacing(np.abs(w)) * 2.0 ** 13   # one TF32 ulp at each value's exponent
    assert np.all(np.abs(r.astype(np.float64) - w) <= ulp / 2)
    np.testing.assert_array_equal(cblib.round_weights_tf32(r), r)
    # ties: 1 + k*2^-10 + 2^-11 rounds to the even k
    base = np.float32(1.0).view(np.uint32)
    tie_even = np.array([base + 0x1000], np.uint32).view(np.float32)        # k = 0 -> 1.0
    tie_odd = np.array([base + 0x2000 + 0x1000], np.uint32).view(np.float32)  # k = 1 -> k = 2
    assert cblib.round_weights_tf32(tie_even)[0] == 1.0
    assert cblib.round_weights_tf32(tie_odd).view(np.uint32)[0] == base + 0x4000
    assert np.isinf(cblib.round_weights_tf32(np.array([np.inf], np.float32))[0])


def test_tuning_overrides_are_validated(cblib):
    """cb_set_tuning knows its knobs by name (unknown names are refused) and resets each with NULL."""
    lib = cblib.load()
    for name, value in (("CB_HALO_FORCE", b"cm,2"), ("CB_HALO_FORCE", b"cm192"), ("CB_HALO_FORCE", b"cm192,0,1,3"),
                        ("CB_HALO_FORCE", b"128,0,2"), ("CB_IGEMM_FORCE", b"64,3,0"), ("CB_IGEMM_BLOCKS", b"1"),
                        ("CB_DW_FORCE", b"4,0,2"), ("CB_DW_BLOCK_FORCE", b"0"), ("CB_DEBUG_PLAN", b""),
                        ("CB_STEM_KERNEL", b"cuda"), ("CB_DEBUG_DW_SKIP_ROW", b"1"), ("CB_DEBUG_STAGE_SKIP_X", b"1"),
                        ("CB_TIMEOUT_MS", b"50")):
        assert lib.cb_set_tuning(name.encode(), value) == cblib.OK
        assert lib.cb_set_tuning(name.encode(), None) == cblib.OK
    assert lib.cb_set_tuning(b"CB_NO_SUCH_KNOB", b"1") == cblib.ERR_INVALID_ARG
    assert lib.cb_set_tuning(None, b"1") == cblib.ERR_INVALID_ARG
    with cblib.tuning("CB_DW_BLOCK_FORCE", "1"):
        pass


def test_last_launch_needs_a_launch(cblib):
    """cb_last_launch reports this thread's last kernel; a thread that launched none gets INVALID_ARG."""
    import threading
    out = []
    info = cblib.CbLaunchInfo()
    t = threading.Thread(target=lambda: out.append(cblib.load().cb_last_launch(ctypes.byref(info))))
    t.start()
    t.join()
    assert out == [cblib.ERR_INVALID_ARG]
    assert cblib.load().cb_last_launch(None) == cblib.ERR_INVALID_ARG


def test_autotune_rejects_in_place_residual(cblib):
    """Each tuning launch writes y, so a residual on y would be added again and again: refused before
    anything runs (fake pointers, never dereferenced)."""
    lib = cblib.load()
    T = ctypes.byref
    base = 1 << 20
    x = _view(base, 1, 8, 8, 32)
    y = _view(base + (1 << 16), 1, 8, 8, 32)
    w = s = b = base + (1 << 18)
    assert lib.cb_autotune_conv(T(x), w, s, b, 3, 3, 1, 1, 1, 2, T(y), 2, T(y), None) == cblib.ERR_INVALID_ARG
    assert lib.cb_autotune_conv(T(x), w, s, b, 3, 3, 1, 1, 1, 2, T(y), 1, T(y), None) == cblib.ERR_INVALID_ARG


def test_convert_weights_bf16_rounds_to_nearest_even(cblib):
    """cb_convert_weights_bf16 equals torch's float32 -> bfloat16 conversion bit for bit (round to nearest,
    ties to even), on random values over a wide range, exact ties, infinities and NaN."""
    import torch
    g = np.random.default_rng(5)
    w = (g.standard_normal(20000) * np.exp(g.uniform(-30, 30, 20000))).astype(np.float32)
    base = np.array([1.0, -3.0], np.float32).view(np.uint32)
    ties = np.concatenate([base + 0x8000, base + 0x18000, base + 0x7FFF, base + 0x8001]).view(np.float32)
    special = np.array([np.inf, -np.inf, 0.0, -0.0, 3.4e38, 1e-40], np.float32)
    w = np.concatenate([w, ties, special])
    got = cblib.convert_weights_bf16(w).view(torch.int16).numpy()
    want = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(got, want)
    nan = cblib.convert_weights_bf16(np.array([np.nan], np.float32)).float().numpy()
    assert np.isnan(nan[0])
