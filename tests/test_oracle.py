"""Pins for the CPU oracle, each against something other than the oracle.

Every check here runs on the CPU (no GPU marker).  The oracle follows the
definition of conv_fprop in the cuDNN documentation page "Convolutions"
(section "Convolution Fprop" and its argument list); these tests tie it to
values printed on the pages, to closed forms, to textbook routines
(scipy.signal correlate2d / convolve2d, an int64 matrix product, a float64
library convolution), to algebraic invariants and to brute force on tiny
inputs.  ``test_planted_mistakes_are_caught`` shows that plausible slips in
the C source (a dropped flip, swapped paddings, a wrong stride or dilation
term, an int32 wrap) each fail at least one of these pins.
"""
import itertools
import os
import re
import shutil
import subprocess

import numpy as np
import pytest
import scipy.signal
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _run(x, w, x_layout="NCHW", w_layout="KCRS", **kw):
    xf, xs = synth.place(x, x_layout)
    wf, ws = synth.place(w, w_layout)
    return oracle.conv_fprop(xf, x.shape, xs, wf, w.shape, ws, **kw)


def _rand(seed, shape, lo=-128, hi=127):
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=shape, dtype=np.int64).astype(np.int8)


def _torch_f64(x, w, pre, post, stride, dilation, mode):
    """float64 torch convolution: exact while |acc| < 2^53."""
    xt = torch.from_numpy(x.astype(np.float64))
    wt = torch.from_numpy(w.astype(np.float64))
    if mode == 1:
        wt = torch.flip(wt, dims=[2, 3])
    xt = F.pad(xt, (pre[1], post[1], pre[0], post[0]))
    return F.conv2d(xt, wt, stride=stride, dilation=dilation).numpy().astype(np.int64)


# --------------------------------------------------------------------------
# Values printed on the pages
# --------------------------------------------------------------------------
def _read_golden_shapes():
    rows = []
    with open(os.path.join(GOLDEN, "output_shapes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            rows.append((list(map(int, lhs.split())), list(map(int, rhs.split()))))
    return rows


@pytest.mark.parametrize("row", _read_golden_shapes())
def test_output_size_matches_printed_shapes(row):
    (N, C, H, W, K, R, S, sh, sw, ph, pw, qh, qw, dh, dw), (P, Q) = row
    assert oracle.out_dims((N, C, H, W), (K, C, R, S), (ph, pw), (qh, qw), (sh, sw), (dh, dw)) == (N, K, P, Q)
    x = _rand(1, (N, C, H, W))
    w = _rand(2, (K, C, R, S))
    y = _run(x, w, pre=(ph, pw), post=(qh, qw), stride=(sh, sw), dilation=(dh, dw))
    assert y.shape == (N, K, P, Q)


def test_forum_words_are_saturated_truth_packed():
    """The forum thread's cuDNN words are its int32 truth clamped to int8 and
    packed four to a little-endian int32 word (the remaining words untouched)."""
    vals = {}
    with open(os.path.join(GOLDEN, "forum_int8_example.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *nums = line.split()
            vals[key] = np.array(list(map(int, nums)), dtype=np.int64)
    words = oracle.pack_int8_words(oracle.saturate_int8(vals["truth"]))
    assert list(words) == list(vals["cudnn"][: len(words)])
    assert np.all(vals["cudnn"][len(words):] == 0)
    # and the int32 truth itself is not what was printed
    assert not np.array_equal(vals["truth"], vals["cudnn"])


def test_forum_descriptor_strides_of_unit_dims_do_not_matter():
    """The forum thread declares X strides [25,1,5,1] and is told to use
    [25,25,5,1]; with C=1 the channel stride is never multiplied by a non-zero
    index, so both describe the same bytes and give the same result."""
    x = _rand(3, (1, 1, 5, 5))
    w = _rand(4, (1, 1, 3, 3))
    xf = x.reshape(-1)
    wf = w.reshape(-1)
    ya = oracle.conv_fprop(xf, x.shape, (25, 1, 5, 1), wf, w.shape, (9, 1, 3, 1))
    yb = oracle.conv_fprop(xf, x.shape, (25, 25, 5, 1), wf, w.shape, (9, 9, 3, 1))
    assert np.array_equal(ya, yb)
    assert ya.shape == (1, 1, 3, 3)


# --------------------------------------------------------------------------
# Brute force and independent library routines
# --------------------------------------------------------------------------
def _small_cases():
    rng = np.random.default_rng(1234)
    cases = []
    for i in range(40):
        R, S = int(rng.integers(1, 4)), int(rng.integers(1, 4))
        sh, sw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        dh, dw = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        pre = (int(rng.integers(0, 3)), int(rng.integers(0, 3)))
        post = (int(rng.integers(0, 3)), int(rng.integers(0, 3)))
        H = int(rng.integers(dh * (R - 1) + 1, 7)) if dh * (R - 1) + 1 < 7 else dh * (R - 1) + 1
        W = int(rng.integers(dw * (S - 1) + 1, 7)) if dw * (S - 1) + 1 < 7 else dw * (S - 1) + 1
        N, C, K = int(rng.integers(1, 3)), int(rng.integers(1, 3)), int(rng.integers(1, 3))
        cases.append(dict(N=N, C=C, H=H, W=W, K=K, R=R, S=S, stride=(sh, sw), dilation=(dh, dw),
                          pre=pre, post=post, mode=i % 2, seed=i))
    return cases


@pytest.mark.parametrize("case", _small_cases())
def test_brute_force_and_float64_library_agree(case):
    c = case
    x = _rand(c["seed"], (c["N"], c["C"], c["H"], c["W"]))
    w = _rand(c["seed"] + 1000, (c["K"], c["C"], c["R"], c["S"]))
    kw = dict(pre=c["pre"], post=c["post"], stride=c["stride"], dilation=c["dilation"], mode=c["mode"])
    y = _run(x, w, **kw)
    assert np.array_equal(y, oracle.conv_fprop_pyint(x, w, **kw))
    assert np.array_equal(y, _torch_f64(x, w, c["pre"], c["post"], c["stride"], c["dilation"], c["mode"]))


@pytest.mark.parametrize("mode", [0, 1])
def test_textbook_correlate_and_convolve(mode):
    """Stride 1, dilation 1, no padding: per output channel, the sum over input
    channels of scipy's 'valid' 2-D cross-correlation (mode 0) or true 2-D
    convolution (mode 1, the kernel rotated by 180 degrees)."""
    x = _rand(10 + mode, (2, 3, 9, 8))
    w = _rand(20 + mode, (4, 3, 3, 2))
    y = _run(x, w, mode=mode)
    op = scipy.signal.correlate2d if mode == 0 else scipy.signal.convolve2d
    ref = np.zeros_like(y, dtype=np.int64)
    for n in range(2):
        for k in range(4):
            for c in range(3):
                ref[n, k] += op(x[n, c].astype(np.int64), w[k, c].astype(np.int64), mode="valid")
    assert np.array_equal(y, ref)


def test_textbook_padding_is_zeros_before_and_after():
    """pre/post padding: scipy 'valid' correlation of the explicitly zero-padded
    image (pre rows/cols before index 0, post after the last)."""
    x = _rand(30, (1, 2, 7, 6))
    w = _rand(31, (3, 2, 3, 3))
    pre, post = (2, 0), (1, 3)
    y = _run(x, w, pre=pre, post=post)
    xp = np.pad(x.astype(np.int64), ((0, 0), (0, 0), (pre[0], post[0]), (pre[1], post[1])))
    ref = np.zeros_like(y, dtype=np.int64)
    for k in range(3):
        for c in range(2):
            ref[0, k] += scipy.signal.correlate2d(xp[0, c], w[k, c].astype(np.int64), mode="valid")
    assert np.array_equal(y, ref)


def test_stride_and_dilation_via_unfold_and_matmul():
    """Explicit im2col (numpy slicing of the zero-padded image) times the
    filter matrix, int64; independent of the oracle's index formula."""
    x = _rand(40, (2, 5, 13, 11))
    w = _rand(41, (6, 5, 3, 2))
    pre, post, stride, dil = (3, 1), (2, 2), (2, 3), (3, 2)
    y = _run(x, w, pre=pre, post=post, stride=stride, dilation=dil)
    xp = np.pad(x.astype(np.int64), ((0, 0), (0, 0), (pre[0], post[0]), (pre[1], post[1])))
    _, _, P, Q = y.shape
    cols = []
    for r in range(3):
        for s in range(2):
            sl = xp[:, :, r * dil[0]: r * dil[0] + stride[0] * (P - 1) + 1: stride[0],
                    s * dil[1]: s * dil[1] + stride[1] * (Q - 1) + 1: stride[1]]
            cols.append(sl)  # [N, C, P, Q] for tap (r, s)
    A = np.stack(cols, axis=2)  # [N, C, R*S, P, Q]
    ref = np.einsum("ncipq,kci->nkpq", A, w.reshape(6, 5, 6).astype(np.int64))
    assert np.array_equal(y, ref)


def test_one_by_one_is_integer_gemm():
    """A 1x1 filter with stride 1 and no padding is Xmat[NHW x C] @ W[K x C]^T."""
    x = _rand(50, (3, 7, 5, 4))
    w = _rand(51, (9, 7, 1, 1))
    xf, xs = synth.place(x, "NHWC")
    wf, ws = synth.place(w, "KRSC")
    yd = (3, 9, 5, 4)
    ystr = synth.packed_strides(yd, "NHWC")
    y = oracle.conv_fprop(xf, x.shape, xs, wf, w.shape, ws, y_strides=ystr)
    ref = xf.reshape(-1, 7).astype(np.int64) @ wf.reshape(9, 7).astype(np.int64).T
    assert np.array_equal(y.reshape(-1, 9), ref)


# --------------------------------------------------------------------------
# Closed forms
# --------------------------------------------------------------------------
def _inbound_taps(size, out, taps, pre, stride, dil):
    """Closed form count of taps r in [0, taps) with 0 <= o*stride - pre + r*dil < size."""
    counts = []
    for o in range(out):
        start = o * stride - pre
        rmin = 0 if start >= 0 else (-start + dil - 1) // dil
        rmax = min(taps - 1, (size - 1 - start) // dil) if size - 1 - start >= 0 else -1
        counts.append(max(0, rmax - rmin + 1))
    return np.array(counts, dtype=np.int64)


@pytest.mark.parametrize("val", [1, -128, 127])
def test_constant_inputs_count_inbound_taps(val):
    N, C, H, W, K, R, S = 2, 3, 9, 7, 2, 4, 3
    pre, post, stride, dil = (3, 2), (2, 4), (2, 1), (2, 3)
    x = np.full((N, C, H, W), val, dtype=np.int8)
    w = np.full((K, C, R, S), -128 if val != 1 else 1, dtype=np.int8)
    y = _run(x, w, pre=pre, post=post, stride=stride, dilation=dil)
    _, _, P, Q = y.shape
    ch = _inbound_taps(H, P, R, pre[0], stride[0], dil[0])
    cw = _inbound_taps(W, Q, S, pre[1], stride[1], dil[1])
    per = int(val) * int(w.flat[0])
    expect = C * per * np.outer(ch, cw)
    for n in range(N):
        for k in range(K):
            assert np.array_equal(y[n, k], expect)


def test_interior_worst_case_reaches_bound():
    """All -128 operands: interior outputs of a 3x3/pad-1 layer equal C*R*S*2^14."""
    C = 40
    x = np.full((1, C, 6, 6), -128, dtype=np.int8)
    w = np.full((2, C, 3, 3), -128, dtype=np.int8)
    y = _run(x, w, pre=(1, 1), post=(1, 1))
    assert y[0, 0, 2, 2] == oracle.worst_case_abs(C, 3, 3) == C * 9 * 16384


def test_accumulator_beyond_int32_is_reported():
    C = 131072 // 16 + 1  # C*R*S*2^14 > 2^31 - 1 with R*S = 16
    x = np.full((1, C, 4, 4), -128, dtype=np.int8)
    w = np.full((1, C, 4, 4), -128, dtype=np.int8)
    with pytest.raises(OverflowError):
        _run(x, w)
    assert oracle.worst_case_abs(C, 4, 4) > 2 ** 31 - 1


def test_config_bounds_fit_int32():
    for cfg in synth.CONFIGS.values():
        bound = oracle.worst_case_abs(cfg.C, cfg.R, cfg.S, (1 << 20) if cfg.bias else 0)
        assert bound <= 2 ** 31 - 1
    assert oracle.worst_case_abs(256, 3, 3) == 37748736


# --------------------------------------------------------------------------
# Invariants
# --------------------------------------------------------------------------
def test_flip_equivalence_between_modes():
    x = _rand(60, (2, 3, 10, 9))
    w = _rand(61, (4, 3, 3, 4))
    kw = dict(pre=(1, 2), post=(2, 0), stride=(2, 1), dilation=(1, 2))
    y_conv = _run(x, w, mode=1, **kw)
    y_flip = _run(x, np.ascontiguousarray(w[:, :, ::-1, ::-1]), mode=0, **kw)
    assert np.array_equal(y_conv, y_flip)
    assert not np.array_equal(y_conv, _run(x, w, mode=0, **kw))


@pytest.mark.parametrize("mode", [0, 1])
def test_impulse_response(mode):
    """A one-hot image at (h0, w0): cross-correlation reads the filter
    backwards across the output, convolution reads it forwards."""
    R, S = 3, 4
    x = np.zeros((1, 1, 12, 12), dtype=np.int8)
    h0, w0 = 6, 5
    x[0, 0, h0, w0] = 1
    w = _rand(62, (1, 1, R, S))
    y = _run(x, w, mode=mode)
    for p in range(y.shape[2]):
        for q in range(y.shape[3]):
            r, s = h0 - p, w0 - q
            if 0 <= r < R and 0 <= s < S:
                exp = w[0, 0, r, s] if mode == 0 else w[0, 0, R - 1 - r, S - 1 - s]
            else:
                exp = 0
            assert y[0, 0, p, q] == exp


def test_linearity_in_image_and_filter():
    kw = dict(pre=(1, 0), post=(0, 1), stride=(1, 2), dilation=(2, 1), mode=1)
    x1, x2 = _rand(70, (2, 4, 8, 8), -64, 63), _rand(71, (2, 4, 8, 8), -64, 63)
    w1, w2 = _rand(72, (3, 4, 3, 2), -64, 63), _rand(73, (3, 4, 3, 2), -64, 63)
    y = _run((x1 + x2).astype(np.int8), w1, **kw).astype(np.int64)
    assert np.array_equal(y, _run(x1, w1, **kw).astype(np.int64) + _run(x2, w1, **kw))
    y = _run(x1, (w1 + w2).astype(np.int8), **kw).astype(np.int64)
    assert np.array_equal(y, _run(x1, w1, **kw).astype(np.int64) + _run(x1, w2, **kw))


def test_shift_equivariance():
    x = _rand(80, (1, 2, 8, 10))
    w = _rand(81, (2, 2, 3, 3))
    xs = np.zeros_like(x)
    xs[..., 1:] = x[..., :-1]
    y, ys = _run(x, w), _run(xs, w)
    assert np.array_equal(ys[..., 1:], y[..., :-1])


@pytest.mark.parametrize("xl,wl", [("NCHW", "KCRS"), ("NHWC", "KRSC"), ("NHWC", "KCRS")])
def test_layout_independence(xl, wl):
    x = _rand(90, (2, 5, 7, 6))
    w = _rand(91, (3, 5, 2, 3))
    kw = dict(pre=(1, 1), post=(0, 1), stride=(1, 2))
    base = _run(x, w, **kw)
    xf, xs = synth.place(x, xl, pad_elems=3)
    wf, ws = synth.place(w, wl, pad_elems=1)
    assert np.array_equal(oracle.conv_fprop(xf, x.shape, xs, wf, w.shape, ws, **kw), base)
    yd = base.shape
    for yl in ("NCHW", "NHWC"):
        ystr = synth.packed_strides(yd, yl)
        yflat = oracle.conv_fprop(xf, x.shape, xs, wf, w.shape, ws, y_strides=ystr, **kw)
        assert np.array_equal(synth.gather_logical(yflat, yd, ystr), base)


def test_bias_then_relu():
    x = _rand(100, (1, 3, 6, 6))
    w = _rand(101, (4, 3, 3, 3))
    b = np.array([-(1 << 20), -5, 0, 1 << 20], dtype=np.int32)
    y0 = _run(x, w).astype(np.int64)
    yb = _run(x, w, bias=b)
    yr = _run(x, w, bias=b, relu=True)
    assert np.array_equal(yb, y0 + b[None, :, None, None])
    assert np.array_equal(yr, np.maximum(y0 + b[None, :, None, None], 0))
    assert np.all(yr[0, 0][y0[0, 0] < (1 << 20)] == 0)


def test_bias_wraps_as_int32():
    x = np.full((1, 1, 1, 1), 127, dtype=np.int8)
    w = np.full((1, 1, 1, 1), 127, dtype=np.int8)
    b = np.array([2 ** 31 - 1], dtype=np.int32)
    y = _run(x, w, bias=b)
    assert y[0, 0, 0, 0] == ((127 * 127 + 2 ** 31 - 1 + 2 ** 31) % 2 ** 32) - 2 ** 31


@pytest.mark.parametrize("shift", [0, 1, 5, 9, 14, 31])
def test_int8_output_is_requantised_int32(shift):
    """int8 output = saturate(floor((y + 2^(shift-1)) / 2^shift)) of the int32
    result, computed here in numpy int64 from the oracle's int32 output."""
    x = _rand(110 + shift, (2, 5, 7, 6))
    w = _rand(111 + shift, (4, 5, 3, 2))
    b = np.array([-(1 << 20), 77, 0, 1 << 19], dtype=np.int32)
    kw = dict(pre=(1, 0), post=(0, 1), stride=(1, 2), bias=b, relu=shift % 2 == 1)
    y32 = _run(x, w, **kw).astype(np.int64)
    y8 = _run(x, w, out_int8=True, out_shift=shift, **kw)
    assert y8.dtype == np.int8
    t = y32 if shift == 0 else np.floor_divide(y32 + (1 << (shift - 1)), 1 << shift)
    assert np.array_equal(y8, np.clip(t, -128, 127))
    if shift == 0:
        assert np.array_equal(y8, oracle.saturate_int8(y32))


def test_int8_output_rounding_and_saturation_closed_forms():
    """A 1x1, one-channel convolution is a product x*w; the rounding right
    shift rounds halves up (towards +inf) and the result saturates."""
    xs = np.array([3, -3, 2, -2, 5, -5, 1, -1, 127, -128, 127], dtype=np.int8)
    ws = np.array([1, 1, 1, 1, 1, 1, 1, 1, 127, 127, -128], dtype=np.int8)
    expect = {0: [3, -3, 2, -2, 5, -5, 1, -1, 127, -128, -128],
              1: [2, -1, 1, -1, 3, -2, 1, 0, 127, -128, -128],
              2: [1, -1, 1, 0, 1, -1, 0, 0, 127, -128, -128],
              8: [0, 0, 0, 0, 0, 0, 0, 0, 63, -63, -63]}
    x = xs.reshape(1, 1, 1, -1)
    for shift, exp in expect.items():
        got = [int(_run(x[..., i:i + 1], ws[i].reshape(1, 1, 1, 1), out_int8=True, out_shift=shift)[0, 0, 0, 0])
               for i in range(len(xs))]
        assert got == exp, (shift, got)


def test_points_match_full_output():
    cfg = synth.CONFIGS["p4_shape"]
    x, w, _ = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    y = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws)
    rng = np.random.default_rng(5)
    pts = np.stack([rng.integers(0, d, 200) for d in y.shape], axis=1)
    vals = oracle.conv_fprop_points(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, pts)
    assert np.array_equal(vals, y[tuple(pts.T)])


def test_generator_is_layout_free_and_seeded():
    a = synth.int8_uniform(7, synth.TAG_X, (2, 3, 4, 5))
    b = synth.int8_uniform(7, synth.TAG_X, (2, 3, 4, 5))
    assert np.array_equal(a, b)
    big = synth.int8_uniform(9, synth.TAG_X, (1 << 16,))
    assert big.min() == -128 and big.max() == 127
    e = synth.int8_with_extremes(11, synth.TAG_X, (1 << 16,), 0.1)
    frac = np.mean((e == -128) | (e == 127))
    assert 0.09 < frac < 0.12
    # published splitmix64 finaliser on a known state (seed 0 stream, first
    # output = mix(0x9E3779B97F4A7C15)): 0xE220A8397B1DCDAF
    assert int(synth.splitmix64(0, 1)[0]) == 0xE220A8397B1DCDAF


# --------------------------------------------------------------------------
# Planted mistakes: each one must break at least one pin above
# --------------------------------------------------------------------------
# ------------------------------------------------------------------ data and weight gradients
# Pins of oracle_conv_dgrad / oracle_conv_wgrad ("Convolutions", sections
# "Convolution Dgrad" and "Convolution Wgrad": the gradients of a loss with
# respect to the image and to the filter, given the loss gradient dY).


def _grads(x, w, dy, pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode=0, layouts=("NCHW", "KCRS")):
    xf, xs = synth.place(x, layouts[0])
    wf, ws = synth.place(w, layouts[1])
    yf, ys = synth.place(dy, layouts[0])
    kw = dict(pre=pre, post=post, stride=stride, dilation=dilation, mode=mode)
    dx = oracle.conv_dgrad(yf, dy.shape, ys, wf, w.shape, ws, x.shape, **kw)
    dw = oracle.conv_wgrad(xf, x.shape, xs, yf, dy.shape, ys, w.shape, **kw)
    return dx, dw


def _grad_case(c):
    x = _rand(c["seed"], (c["N"], c["C"], c["H"], c["W"]))
    w = _rand(c["seed"] + 1000, (c["K"], c["C"], c["R"], c["S"]))
    kw = dict(pre=c["pre"], post=c["post"], stride=c["stride"], dilation=c["dilation"], mode=c["mode"])
    yd = oracle.out_dims(x.shape, w.shape, c["pre"], c["post"], c["stride"], c["dilation"])
    dy = _rand(c["seed"] + 2000, yd)
    return x, w, dy, kw


@pytest.mark.parametrize("case", _small_cases()[:20])
def test_grads_are_the_adjoints_of_fprop(case):
    """fprop is bilinear, so for every X, W, dY:
    <fprop(X, W), dY> = <X, dgrad(dY, W)> = <W, wgrad(X, dY)>  (exact integers).
    Ties both gradients to the pinned forward oracle."""
    x, w, dy, kw = _grad_case(case)
    y = _run(x, w, **kw).astype(np.int64)
    dx, dw = _grads(x, w, dy, **kw)
    lhs = int((y * dy.astype(np.int64)).sum())
    assert lhs == int((x.astype(np.int64) * dx.astype(np.int64)).sum())
    assert lhs == int((w.astype(np.int64) * dw.astype(np.int64)).sum())


@pytest.mark.parametrize("case", _small_cases()[20:32])
def test_grads_brute_force_chain_rule(case):
    """Element by element against the chain rule applied term by term to the
    forward definition (Python integers, scatter order)."""
    x, w, dy, kw = _grad_case(case)
    dx, dw = _grads(x, w, dy, **kw)
    px, pw = oracle.grads_pyint(x, w, dy, **kw)
    assert np.array_equal(dx, px)
    assert np.array_equal(dw, pw)


@pytest.mark.parametrize("case", _small_cases()[32:40])
def test_grads_match_float64_autograd(case):
    """Element by element against PyTorch autograd of a float64 conv2d (exact:
    every value is an integer far below 2^53); convolution mode flips the
    filter before the library's cross-correlation."""
    x, w, dy, kw = _grad_case(case)
    dx, dw = _grads(x, w, dy, **kw)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    pre, post = kw["pre"], kw["post"]
    xp = F.pad(xt, (pre[1], post[1], pre[0], post[0]))
    weff = torch.flip(wt, [2, 3]) if kw["mode"] else wt
    y = F.conv2d(xp, weff, stride=kw["stride"], dilation=kw["dilation"])
    assert tuple(y.shape) == dy.shape
    (y * torch.tensor(dy, dtype=torch.float64)).sum().backward()
    assert np.array_equal(dx, xt.grad.numpy().astype(np.int64))
    assert np.array_equal(dw, wt.grad.numpy().astype(np.int64))


def test_grads_one_by_one_are_integer_gemms():
    """1x1 filter, stride 1, no padding: dX[n,:,h,w] = W^T dY[n,:,h,w] and
    dW = sum over pixels of dY x X^T (int64 matrix products)."""
    x = _rand(60, (2, 5, 4, 3))
    w = _rand(61, (6, 5, 1, 1))
    dy = _rand(62, (2, 6, 4, 3))
    dx, dw = _grads(x, w, dy, layouts=("NHWC", "KRSC"))
    wm = w[:, :, 0, 0].astype(np.int64)                      # K x C
    ym = dy.transpose(0, 2, 3, 1).reshape(-1, 6).astype(np.int64)  # pixels x K
    xm = x.transpose(0, 2, 3, 1).reshape(-1, 5).astype(np.int64)   # pixels x C
    assert np.array_equal(dx.transpose(0, 2, 3, 1).reshape(-1, 5), ym @ wm)
    assert np.array_equal(dw[:, :, 0, 0], ym.T @ xm)


def test_dgrad_stride_two_leaves_unreached_pixels_zero():
    """Stride 2, 1x1 filter, no padding: only pixels on the stride grid feed the
    output, so every other row and column of dX is zero and the grid holds
    W^T dY."""
    x = np.zeros((1, 2, 6, 6), dtype=np.int8)
    w = _rand(63, (3, 2, 1, 1))
    dy = _rand(64, (1, 3, 3, 3))
    dx, _ = _grads(x, w, dy, stride=(2, 2))
    assert np.all(dx[:, :, 1::2, :] == 0) and np.all(dx[:, :, :, 1::2] == 0)
    ref = np.einsum("kc,nkpq->ncpq", w[:, :, 0, 0].astype(np.int64), dy.astype(np.int64))
    assert np.array_equal(dx[:, :, ::2, ::2], ref)


def test_wgrad_accumulator_bound():
    """dW sums N*P*Q products of two int8 values: an all-(-128) image and loss
    gradient over 131072 pixels reach 2^31 and are reported, one pixel fewer
    fits int32."""
    x = np.full((1, 1, 256, 512), -128, dtype=np.int8)
    dy = np.full((1, 1, 256, 512), -128, dtype=np.int8)
    with pytest.raises(OverflowError):
        oracle.conv_wgrad(x.ravel(), x.shape, (131072, 131072, 512, 1), dy.ravel(), dy.shape,
                          (131072, 131072, 512, 1), (1, 1, 1, 1))
    x2 = x.copy()
    x2[0, 0, 0, 0] = 0
    dw = oracle.conv_wgrad(x2.ravel(), x.shape, (131072, 131072, 512, 1), dy.ravel(), dy.shape,
                           (131072, 131072, 512, 1), (1, 1, 1, 1))
    assert int(dw.ravel()[0]) == 131071 * 16384


MUTATIONS = {
    "no_flip": ("int64_t rf = pp->mode ? (R - 1 - r) : r;", "int64_t rf = r;"),
    "pre_post_swapped": ("int64_t h = p * pp->stride[0] - pp->pre[0] + r * pp->dil[0];",
                         "int64_t h = p * pp->stride[0] - pp->post[0] + r * pp->dil[0];"),
    "dilation_dropped": ("int64_t ww = q * pp->stride[1] - pp->pre[1] + s * pp->dil[1];",
                         "int64_t ww = q * pp->stride[1] - pp->pre[1] + s;"),
    "filter_k_uses_c_stride": ("int64_t wv = w[k * ws[0] +", "int64_t wv = w[k * ws[1] +"),
    "padding_not_zero": ("continue; /* zero padding */", "{ h = h < 0 ? 0 : (h >= H ? H - 1 : h); ww = ww < 0 ? 0 : (ww >= W ? W - 1 : ww); }"),
    "relu_before_bias": ("if (bias) v = (int32_t)((uint32_t)v + (uint32_t)bias[k]);\n    if (pp->relu && v < 0) v = 0;",
                         "if (pp->relu && v < 0) v = 0;\n    if (bias) v = (int32_t)((uint32_t)v + (uint32_t)bias[k]);"),
    "int8_no_saturation": ("    if (t > 127) t = 127;\n", ""),
    "int8_truncating_shift": ("        t += (int64_t)1 << (shift - 1);\n", ""),
    "dgrad_floor_instead_of_exact_division": ("if (th < 0 || th % pp->stride[0]) continue;", "if (th < 0) continue;"),
    "dgrad_filter_not_flipped": ("int64_t wv = w[k * ws[0] + c * ws[1] + rf * ws[2] + sf * ws[3]];\n                                acc += gv * wv;",
                                 "int64_t wv = w[k * ws[0] + c * ws[1] + r * ws[2] + s * ws[3]];\n                                acc += gv * wv;"),
    "dgrad_post_for_pre": ("int64_t tw = ww + pp->pre[1] - s * pp->dil[1];", "int64_t tw = ww + pp->post[1] - s * pp->dil[1];"),
    "wgrad_output_not_flipped": ("dw[k * ws[0] + c * ws[1] + rf * ws[2] + sf * ws[3]] = (int32_t)acc;",
                                 "dw[k * ws[0] + c * ws[1] + r * ws[2] + s * ws[3]] = (int32_t)acc;"),
    "wgrad_loss_index_uses_image_channel": ("int64_t gv = dy[n * ys[0] + k * ys[1] + p * ys[2] + q * ys[3]];\n                                int64_t xv",
                                            "int64_t gv = dy[n * ys[0] + (c % K) * ys[1] + p * ys[2] + q * ys[3]];\n                                int64_t xv"),
}

_PIN_FUNCS = None


def _pin_suite():
    """Run the pins as plain functions; return True when all pass."""
    funcs = [
        lambda: [test_brute_force_and_float64_library_agree(c) for c in _small_cases()[:12]],
        lambda: [test_textbook_correlate_and_convolve(m) for m in (0, 1)],
        test_textbook_padding_is_zeros_before_and_after,
        test_stride_and_dilation_via_unfold_and_matmul,
        test_one_by_one_is_integer_gemm,
        lambda: [test_constant_inputs_count_inbound_taps(v) for v in (1, -128)],
        test_flip_equivalence_between_modes,
        test_bias_then_relu,
        test_int8_output_rounding_and_saturation_closed_forms,
        lambda: [test_grads_are_the_adjoints_of_fprop(c) for c in _small_cases()[:12]],
        test_grads_one_by_one_are_integer_gemms,
        test_dgrad_stride_two_leaves_unreached_pixels_zero,
    ]
    for f in funcs:
        try:
            f()
        except AssertionError:
            return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "conv_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", str(mutated), "-o", str(lib)], check=True)
    try:
        oracle.use_library(str(lib))
        assert not _pin_suite(), f"planted mistake {name} survived every pin"
    finally:
        oracle.use_library(None)
