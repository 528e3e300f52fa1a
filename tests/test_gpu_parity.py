"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle,
element by element, bit-exact (integer work: tolerance 0).

Full outputs are compared everywhere; the two largest workloads also at
reduced batch here (same tiling, same code path).  Their full-size outputs,
in the launch configuration the benchmark times, are compared in full in
test_gpu_fullsize.py."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ic():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import int8_conv2d_fprop_gb300 as m
    torch.cuda.set_device(0)
    return m


def _to_dev(flat, dims, strides):
    return torch.as_strided(torch.from_numpy(np.ascontiguousarray(flat)).cuda(), tuple(dims), tuple(strides))


def _run_both(ic, cfg, algo=0, x=None, w=None, b=None, x_pad=0, w_pad=0, y_layout=None, out_shift=None):
    if x is None:
        x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout, pad_elems=x_pad)
    wf, ws = synth.place(w, cfg.w_layout, pad_elems=w_pad)
    xt, wt = _to_dev(xf, cfg.x_dims, xs), _to_dev(wf, cfg.w_dims, ws)
    bt = torch.from_numpy(b).cuda() if b is not None else None
    yl = y_layout or cfg.y_layout
    fmt = torch.channels_last if yl == "NHWC" else torch.contiguous_format
    # canaries around the output: 64 guard words on each side
    P, Q = cfg.P, cfg.Q
    ysz = cfg.N * cfg.K * P * Q
    fill = 0x5A5A5A5A if out_shift is None else 0x5A
    guard = torch.full((ysz + 128,), fill, dtype=torch.int32 if out_shift is None else torch.int8, device="cuda")
    ystr = synth.packed_strides(cfg.y_dims, yl)
    yt = torch.as_strided(guard[64:64 + ysz], cfg.y_dims, ystr)
    y = ic.conv_fprop(xt, wt, bt, pre_padding=cfg.pre, post_padding=cfg.post, stride=cfg.stride,
                      dilation=cfg.dilation, mode=cfg.mode, relu=cfg.relu, algo=algo, out=yt, out_shift=out_shift)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    g = guard.cpu().numpy()
    assert np.all(g[:64] == fill) and np.all(g[64 + ysz:] == fill), "write outside the output"
    got = y.cpu().numpy()
    if out_shift is not None:
        ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                                cfg.dilation, cfg.mode, b, cfg.relu, out_int8=True, out_shift=out_shift)
        return got, ref
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, b, cfg.relu)
    return got, ref


def _assert_equal(got, ref, what):
    if not np.array_equal(got, ref):
        idx = np.argwhere(got != ref)
        first = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {ref.size} outputs differ; first at {first}: "
                             f"got {got[first]} expected {ref[first]}")


# ------------------------------------------------------------------ workloads
@pytest.mark.parametrize("name", ["c1_tiny_nchw", "p4_shape", "c2_s2_nhwc", "c4_1x1_bias_relu"])
def test_workload_full(ic, name):
    cfg = synth.CONFIGS[name]
    got, ref = _run_both(ic, cfg)
    _assert_equal(got, ref, name)


@pytest.mark.parametrize("name,batch", [("c3_3x3_large", 2), ("c5_7x1_dilated_conv", 2)])
def test_workload_reduced_batch_full(ic, name, batch):
    import dataclasses
    cfg = dataclasses.replace(synth.CONFIGS[name], N=batch)
    got, ref = _run_both(ic, cfg)
    _assert_equal(got, ref, f"{name} N={batch}")


# ------------------------------------------------------------------ every algorithm
ALGOS = [1, 2, 3, 4]  # implicit GEMM (TMA im2col), dp4a, generic, implicit GEMM (global loads)


def _shape_cases():
    C = synth.ConvConfig
    return [
        C("ragged_m_k", 3, 64, 13, 11, 200, 3, 3, pre=(1, 1), post=(1, 1), seed=11),
        C("c80_masked", 2, 80, 9, 9, 72, 3, 2, stride=(2, 1), pre=(1, 0), post=(0, 1), seed=12),
        C("c48_single_step", 2, 48, 10, 7, 40, 2, 2, dilation=(2, 3), pre=(2, 2), post=(1, 3), seed=13),
        C("c24_repacked", 2, 24, 8, 8, 36, 3, 3, pre=(1, 1), post=(1, 1), mode=1, bias=True, relu=True, seed=14),
        C("nchw_conv_mode", 2, 32, 11, 12, 20, 4, 2, stride=(1, 2), dilation=(2, 1), pre=(3, 0), post=(2, 1),
          mode=1, x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=15),
        C("one_by_one_strided", 2, 128, 15, 15, 130, 1, 1, stride=(2, 2), bias=True, seed=16),
        C("tiny_c3", 1, 3, 12, 9, 10, 3, 3, pre=(1, 1), post=(1, 1), x_layout="NCHW", w_layout="KCRS",
          y_layout="NCHW", seed=17),
        # 129..192 output channels: 192-column tiles, ragged K
        C("k150_nt192", 2, 96, 9, 11, 150, 3, 3, stride=(1, 2), pre=(1, 1), post=(1, 0), bias=True, seed=18),
        # NCHW images whose H stride and dilation share a factor: the
        # channels-last copy keeps only the rows the windows read (odd rows
        # here: pre-padding 1; W = 13 takes the generic copy)
        C("rows_odd_generic", 2, 40, 21, 13, 72, 3, 3, stride=(2, 1), dilation=(2, 1), pre=(1, 1), post=(2, 1),
          x_layout="NCHW", w_layout="KCRS", seed=19),
        # every third row from row 1 (gcd 3), plane copy (W = 32), convolution mode
        C("rows_gcd3_planes", 2, 32, 30, 32, 64, 5, 3, stride=(3, 1), dilation=(3, 2), pre=(2, 1), post=(3, 1),
          mode=1, x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=20),
        # a 1x1 filter at stride 2: every other row
        C("rows_1x1_s2", 2, 48, 15, 16, 40, 1, 1, stride=(2, 2), x_layout="NCHW", w_layout="KCRS", seed=21),
        # pointwise over dense channels-last rows (2-D pixel-row boxes): 80
        # channels (the second k-step's box runs past a pixel's channels), a
        # partial last tile of 61 pixels
        C("pointwise_c80_ragged", 3, 80, 7, 9, 100, 1, 1, bias=True, relu=True, seed=22),
    ]


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", _shape_cases(), ids=lambda c: c.name)
def test_algorithms_agree_with_oracle(ic, case, algo):
    if algo == 2 and case.C * case.R * case.S > 1024:
        pytest.skip("dp4a takes C*R*S <= 1024")
    got, ref = _run_both(ic, case, algo=algo)
    _assert_equal(got, ref, f"{case.name} algo {algo}")


def _int8_out_cases():
    C = synth.ConvConfig
    return [
        # NHWC, K % 16 == 0: the tensor-core path writes through TMA tensor stores
        C("nhwc_k64", 3, 64, 13, 11, 64, 3, 3, pre=(1, 1), post=(1, 1), bias=True, seed=41),
        # ragged K (not a multiple of 16): plain byte stores
        C("nhwc_ragged_k", 2, 80, 9, 9, 200, 3, 2, stride=(2, 1), pre=(1, 0), post=(0, 1), relu=True, seed=42),
        C("nchw_conv_mode", 2, 32, 11, 12, 20, 4, 2, stride=(1, 2), dilation=(2, 1), pre=(3, 0), post=(2, 1),
          mode=1, bias=True, relu=True, x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=43),
        C("one_by_one_k256", 2, 128, 15, 15, 256, 1, 1, stride=(2, 2), bias=True, seed=44),
        # 192-column tiles write int8 with plain stores (96 columns per epilogue warp)
        C("nhwc_k160_nt192", 2, 64, 10, 12, 160, 3, 3, pre=(1, 1), post=(1, 1), bias=True, relu=True, seed=45),
    ]


@pytest.mark.parametrize("shift", [0, 7, 12])
@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("case", _int8_out_cases(), ids=lambda c: c.name)
def test_int8_output_matches_oracle(ic, case, algo, shift):
    """int8 output (rounding right shift, then saturation) on every algorithm;
    shift 0 saturates almost every output, 12 leaves most in range."""
    if algo == 2 and case.C * case.R * case.S > 1024:
        pytest.skip("dp4a takes C*R*S <= 1024")
    got, ref = _run_both(ic, case, algo=algo, out_shift=shift)
    assert got.dtype == np.int8
    _assert_equal(got, ref, f"{case.name} algo {algo} shift {shift}")


def test_int8_output_large_workload_reduced_batch(ic):
    import dataclasses
    cfg = dataclasses.replace(synth.CONFIGS["c3_3x3_large"], N=2)
    got, ref = _run_both(ic, cfg, out_shift=12)
    _assert_equal(got, ref, "c3 N=2 int8 out")
    # a shift that leaves most values inside the int8 range exercises the rounding
    assert np.mean(np.abs(ref.astype(np.int32)) < 127) > 0.5


@pytest.mark.parametrize("algo", ALGOS)
def test_padded_strides_and_output_layouts(ic, algo):
    cfg = synth.ConvConfig("strided", 2, 32, 9, 10, 24, 3, 3, pre=(1, 2), post=(0, 1), seed=21)
    for yl in ("NCHW", "NHWC"):
        got, ref = _run_both(ic, cfg, algo=algo, x_pad=16, w_pad=3, y_layout=yl)
        _assert_equal(got, ref, f"padded strides algo {algo} y {yl}")


@pytest.mark.parametrize("k_pad,n_pad", [(0, 0), (16, 0), (4, 96)])
@pytest.mark.parametrize("case", [
    synth.ConvConfig("pq64_k40_ragged", 3, 48, 8, 8, 40, 3, 3, pre=(1, 1), post=(1, 1), seed=51),
    synth.ConvConfig("pq96_k256_bias_relu", 2, 64, 12, 8, 256, 1, 1, bias=True, relu=True, seed=52),
    synth.ConvConfig("pq32_k130_s2", 5, 32, 8, 16, 130, 3, 3, stride=(2, 2), pre=(1, 1), post=(0, 0), seed=53),
], ids=lambda c: c.name)
def test_channel_major_output(ic, case, k_pad, n_pad):
    """NCHW outputs whose P*Q is a multiple of 32 take the channel-major TMA
    store; channel and image strides padded beyond P*Q and K*ks must be
    honoured, channels past K and images past N clipped, and nothing written
    outside the output (canaries)."""
    cfg = case
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    xt, wt = _to_dev(xf, cfg.x_dims, xs), _to_dev(wf, cfg.w_dims, ws)
    bt = torch.from_numpy(b).cuda() if b is not None else None
    N, K, P, Q = cfg.y_dims
    assert (P * Q) % 32 == 0
    ks = P * Q + k_pad
    ns = K * ks + n_pad
    span = (N - 1) * ns + (K - 1) * ks + P * Q
    fill = 0x5A5A5A5A
    guard = torch.full((span + 128,), fill, dtype=torch.int32, device="cuda")
    yt = torch.as_strided(guard[64:64 + span], (N, K, P, Q), (ns, ks, Q, 1))
    y = ic.conv_fprop(xt, wt, bt, pre_padding=cfg.pre, post_padding=cfg.post, stride=cfg.stride,
                      dilation=cfg.dilation, mode=cfg.mode, relu=cfg.relu, out=yt)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    g = guard.cpu().numpy()
    assert np.all(g[:64] == fill) and np.all(g[64 + span:] == fill), "write outside the output"
    # the padding between channels and between images is left alone
    inside = np.zeros(span, dtype=bool)
    for n in range(N):
        for k in range(K):
            inside[n * ns + k * ks:n * ns + k * ks + P * Q] = True
    assert np.all(g[64:64 + span][~inside] == fill), "write into the stride padding"
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, b, cfg.relu)
    _assert_equal(y.cpu().numpy(), ref, f"{cfg.name} k_pad {k_pad} n_pad {n_pad}")


def _partial_round_cases():
    C = synth.ConvConfig
    return [
        # 196 tiles of 256 channels, 18 k-steps
        C("rounds_3x3_nt256", 8, 128, 56, 56, 256, 3, 3, pre=(1, 1), post=(1, 1), seed=61),
        # 196 tiles of 128 channels, 4 k-steps, bias and ReLU
        C("rounds_1x1_bias_relu", 32, 256, 28, 28, 128, 1, 1, bias=True, relu=True, seed=62),
        # 166 tiles over two channel tiles (K = 300), ragged pixels and channels
        C("rounds_ragged_two_ntiles", 5, 96, 45, 47, 300, 3, 3, pre=(1, 1), post=(1, 1), seed=63),
        # 172 tiles, 72 k-steps: five groups of at most 16 k-steps per tile
        C("rounds_long_reduction", 7, 512, 56, 56, 128, 3, 3, pre=(1, 1), post=(1, 1), seed=64),
        # 168 tiles, NCHW image and output (channel-major stores), convolution mode
        C("rounds_nchw_conv_mode", 4, 64, 86, 64, 192, 7, 1, stride=(1, 1), dilation=(2, 1), pre=(6, 0),
          post=(6, 0), mode=1, x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=65),
    ]


@pytest.mark.parametrize("case", _partial_round_cases(), ids=lambda c: c.name)
def test_more_tiles_than_sms_matches_oracle(ic, case):
    """More tiles than SMs, the last round partial: every CTA walks several
    tiles and some CTAs one more than others.  Every output element is
    compared, twice (a second call on the same workspace)."""
    got, ref = _run_both(ic, case)
    _assert_equal(got, ref, case.name)
    got2, _ = _run_both(ic, case)
    _assert_equal(got2, ref, case.name + " (second call)")


def test_tile_shape_on_the_device(ic):
    """The planner's tiles and work units on this GPU: with 152 SMs the 3x3
    workload's 784 tiles leave a partial sixth round of 24 tiles, each cut
    into 6 runs of its 36 k-steps (760 whole tiles + 144 runs); the other
    workloads run whole tiles."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = {}
    for name in ("c2_s2_nhwc", "c3_3x3_large", "c4_1x1_bias_relu", "c5_7x1_dilated_conv"):
        cfg = synth.CONFIGS[name]
        shapes[name] = ic.tile_shape(ic.TensorDesc.packed(ic.CONV_INT8, cfg.x_dims, cfg.x_layout),
                                     ic.TensorDesc.packed(ic.CONV_INT8, cfg.w_dims, cfg.w_layout),
                                     ic.TensorDesc.packed(ic.CONV_INT32, cfg.y_dims, cfg.y_layout),
                                     ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode,
                                                    cfg.bias, cfg.relu))
    assert shapes["c2_s2_nhwc"] == (128, 128, 49, 49)
    assert shapes["c4_1x1_bias_relu"] == (128, 128, 392, 392)
    assert shapes["c5_7x1_dilated_conv"] == (128, 192, 672, 672)
    if sms == 152:
        assert shapes["c3_3x3_large"] == (128, 256, 784, 760 + 24 * 6)


def test_more_tiles_than_sms_int8_output(ic):
    cfg = _partial_round_cases()[1]
    got, ref = _run_both(ic, cfg, out_shift=14)
    _assert_equal(got, ref, "int8 output, partial last round")


@pytest.mark.parametrize("c_pad,n_pad", [(0, 0), (48, 0), (16, 256)])
@pytest.mark.parametrize("case", [
    synth.ConvConfig("planes_c24_hw144", 3, 24, 9, 16, 40, 3, 3, pre=(1, 1), post=(1, 1), x_layout="NCHW",
                     w_layout="KCRS", seed=71),
    synth.ConvConfig("planes_c80_hw400", 2, 80, 20, 20, 96, 3, 1, stride=(2, 1), pre=(1, 0), post=(1, 0),
                     x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=72),
    synth.ConvConfig("planes_c130_hw512", 2, 130, 16, 32, 64, 1, 1, x_layout="NCHW", w_layout="KCRS", seed=73),
], ids=lambda c: c.name)
def test_nchw_image_plane_copy(ic, case, c_pad, n_pad):
    """Images whose channels each hold a contiguous H x W plane (H*W a
    multiple of 16) are either read in place (whole image rows by TMA, when
    the rows and the windows allow it: the 1x1 case here) or copied to
    channels-last by a shared-memory transpose before the tensor-core
    kernel; channel and image strides padded beyond the plane must be
    honoured."""
    cfg = case
    x, w, b = synth.make_inputs(cfg)
    N, C, H, W = cfg.x_dims
    cs = H * W + c_pad
    ns = C * cs + n_pad
    xflat = np.zeros((N - 1) * ns + (C - 1) * cs + H * W, dtype=np.int8)
    for n in range(N):
        for c in range(C):
            xflat[n * ns + c * cs:n * ns + c * cs + H * W] = x[n, c].reshape(-1)
    xs = (ns, cs, W, 1)
    wf, ws = synth.place(w, cfg.w_layout)
    xt, wt = _to_dev(xflat, cfg.x_dims, xs), _to_dev(wf, cfg.w_dims, ws)
    bt = torch.from_numpy(b).cuda() if b is not None else None
    y = ic.conv_fprop(xt, wt, bt, pre_padding=cfg.pre, post_padding=cfg.post, stride=cfg.stride,
                      dilation=cfg.dilation, mode=cfg.mode, relu=cfg.relu, algo=ic.ALGO_IMPLICIT_GEMM)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    ref = oracle.conv_fprop(xflat, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, b, cfg.relu)
    _assert_equal(y.cpu().numpy(), ref, f"{cfg.name} c_pad {c_pad} n_pad {n_pad}")


def _nchw_rows_cases():
    C = synth.ConvConfig
    return [
        # the 7x1 dilated workload's shape at batch 3: a 128-pixel tile spans
        # two output rows (Q = 96), ragged pixel tail, convolution mode,
        # 192-column tiles, channel-major output
        C("rows_7x1_dilated_conv", 3, 128, 28, 96, 192, 7, 1, stride=(2, 1), dilation=(2, 1), pre=(6, 0),
          post=(5, 0), mode=1, x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=81),
        # 3x3, dilation 4 along W (tap offsets 0, 4, 8 around pre-padding 4),
        # 80 channels (the second channel step half past C), 128-column
        # tiles, pixel-major output, bias and ReLU
        C("rows_3x3_dilw4_c80", 2, 80, 20, 32, 96, 3, 3, dilation=(1, 4), pre=(1, 4), post=(1, 4), bias=True,
          relu=True, x_layout="NCHW", w_layout="KCRS", y_layout="NHWC", seed=82),
        # 16-byte image rows: a tile spans eight output rows
        C("rows_w16_1x3", 4, 64, 12, 16, 128, 1, 3, dilation=(1, 4), pre=(0, 4), post=(0, 4), x_layout="NCHW",
          w_layout="KRSC", y_layout="NCHW", seed=83),
        # five tiles, 70 k-steps: each tile cut into runs whose int32 sums the
        # reduction kernel adds
        C("rows_cut_tiles", 1, 640, 20, 32, 64, 7, 1, pre=(3, 0), post=(3, 0), x_layout="NCHW", w_layout="KCRS",
          y_layout="NHWC", seed=84),
    ]


@pytest.mark.parametrize("case", _nchw_rows_cases(), ids=lambda c: c.name)
def test_nchw_rows_read_in_place(ic, case):
    """NCHW images with rows of at most 192 bytes (a multiple of 16), stride 1
    along W and tap offsets that are multiples of 4 are read in place: each
    k-step loads whole image rows of 64 channels, and the converters
    transpose them into the tensor-memory image stage (pixels permuted within
    each 32-lane quadrant, channels within each 16) with the filter repacked
    in the same channel order.  The call launches no image copy."""
    xd = ic.TensorDesc.make(ic.CONV_INT8, case.x_dims, synth.packed_strides(case.x_dims, case.x_layout),
                            int(np.prod(case.x_dims)))
    wd = ic.TensorDesc.make(ic.CONV_INT8, case.w_dims, synth.packed_strides(case.w_dims, case.w_layout),
                            int(np.prod(case.w_dims)))
    yd = ic.TensorDesc.make(ic.CONV_INT32, case.y_dims, synth.packed_strides(case.y_dims, case.y_layout),
                            int(np.prod(case.y_dims)) * 4)
    p = ic.Params.make(case.pre, case.post, case.stride, case.dilation, case.mode, case.bias, case.relu)
    # filter repack and convolution (plus the reduction of the cut tiles)
    assert ic.kernel_count(xd, wd, yd, p) == (3 if case.name == "rows_cut_tiles" else 2)
    got, ref = _run_both(ic, case)
    _assert_equal(got, ref, case.name)


def test_nchw_rows_int8_output(ic):
    """The in-place NCHW path with the int8 requantising epilogue, on 128-
    and 192-column tiles."""
    for case in _nchw_rows_cases()[:2]:
        got, ref = _run_both(ic, case, out_shift=10)
        _assert_equal(got, ref, case.name + " int8 out")


def _filter_in_kernel_cases():
    C = synth.ConvConfig
    return [
        # K = 100 (filter rows past K read as zeros), C = 80 (the second
        # channel step half past C), 3x3 pad 1, convolution mode, bias + ReLU,
        # 128-column tiles
        C("selfw_k100_c80_conv", 2, 80, 14, 13, 100, 3, 3, pre=(1, 1), post=(1, 1), mode=1, bias=True, relu=True,
          seed=91),
        # 192-column tiles, stride 2, dilation 2
        C("selfw_k160_s2_dil2", 3, 64, 19, 17, 160, 3, 3, stride=(2, 2), dilation=(2, 2), pre=(2, 2), post=(2, 1),
          seed=92),
        # 1x1 over pixel rows, channel-major output
        C("selfw_1x1_nchw_out", 4, 128, 12, 16, 64, 1, 1, y_layout="NCHW", seed=93),
        # two tiles, 144 k-steps: each tile cut into runs (the reduction
        # kernel adds their int32 sums)
        C("selfw_cut_tiles", 1, 1024, 12, 12, 128, 3, 3, pre=(1, 1), post=(1, 1), seed=94),
        # an NCHW image of 20-byte rows (copied to channels-last first) with a
        # KRSC filter (converted in the kernel)
        C("selfw_nchw_copy", 2, 48, 11, 20, 80, 3, 3, pre=(1, 1), post=(1, 1), x_layout="NCHW", y_layout="NCHW",
          seed=95),
    ]


@pytest.mark.parametrize("w_pad", [0, 16, 3])
@pytest.mark.parametrize("case", _filter_in_kernel_cases(), ids=lambda c: c.name)
def test_filter_converted_in_kernel(ic, case, w_pad):
    """128- and 192-column tiles over a channels-last image convert a filter
    whose channels are contiguous themselves (TMA loads of int8 filter tiles,
    converted beside the image tile): conv_fprop launches the convolution
    alone.  Filter rows padded to a 16-byte multiple keep that path; padded
    to an odd stride they take the repack instead.  Exact either way."""
    if w_pad == 0:
        xd = ic.TensorDesc.packed(ic.CONV_INT8, case.x_dims, case.x_layout)
        wd = ic.TensorDesc.packed(ic.CONV_INT8, case.w_dims, case.w_layout)
        yd = ic.TensorDesc.packed(ic.CONV_INT32, case.y_dims, case.y_layout)
        p = ic.Params.make(case.pre, case.post, case.stride, case.dilation, case.mode, case.bias, case.relu)
        # the convolution (and the reduction of cut tiles, or the image
        # copy before it), no repack
        assert ic.kernel_count(xd, wd, yd, p) == (2 if case.name in ("selfw_cut_tiles", "selfw_nchw_copy") else 1)
    got, ref = _run_both(ic, case, w_pad=w_pad)
    _assert_equal(got, ref, f"{case.name} w_pad {w_pad}")
    got, ref = _run_both(ic, case, w_pad=w_pad, out_shift=9)
    _assert_equal(got, ref, f"{case.name} w_pad {w_pad} int8 out")


def test_filter_in_kernel_unaligned_pointer_and_prepacked(ic):
    """A filter pointer off the 16-byte grid makes conv_fprop repack the
    filter (another launch-cache key); conv_fprop_pack_filter followed by
    conv_fprop_prepacked reads the repacked blocks, with either pointer.
    All exact."""
    cfg = _filter_in_kernel_cases()[0]
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride, cfg.dilation,
                            cfg.mode, b, cfg.relu)
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))
    yd = ic.TensorDesc.make(ic.CONV_INT32, cfg.y_dims, ystr, ysz * 4)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
    need = ic.workspace_size(xd, wd, yd, p)
    s = torch.cuda.current_stream().cuda_stream
    xt = torch.from_numpy(xf).cuda()
    bt = torch.from_numpy(b).cuda()
    wsb = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
    for off in (0, 8):
        wb = torch.zeros(wf.size + 64, dtype=torch.int8, device="cuda")
        wb[16 + off:16 + off + wf.size].copy_(torch.from_numpy(wf))
        wptr = wb.data_ptr() + 16 + off
        for how in ("conv_fprop", "prepacked"):
            yb = torch.full((ysz,), -1, dtype=torch.int32, device="cuda")
            if how == "conv_fprop":
                st = ic.conv_fprop_raw(xd, xt.data_ptr(), wd, wptr, yd, yb.data_ptr(), bt.data_ptr(), p,
                                       wsb.data_ptr(), need, s)
            else:
                st = ic.pack_filter_raw(xd, wd, wptr, yd, p, wsb.data_ptr(), need, s)
                assert st == 0, ic.STATUS.get(st)
                st = ic.conv_fprop_prepacked_raw(xd, xt.data_ptr(), wd, wptr, yd, yb.data_ptr(), bt.data_ptr(), p,
                                                 wsb.data_ptr(), need, s)
            assert st == 0, ic.STATUS.get(st)
            torch.cuda.synchronize()
            assert ic.device_status() == 0
            got = synth.gather_logical(yb.cpu().numpy(), cfg.y_dims, ystr)
            _assert_equal(got, ref, f"filter offset {off} {how}")


# ------------------------------------------------------------------ exactness
def test_extreme_values_exceed_f32_integer_range(ic):
    """All -128 operands: interior sums C*R*S*2^14 = 37,748,736 > 2^24, so
    the f16 tensor path is exact only through its int32 group sums."""
    cfg = synth.ConvConfig("all_min", 1, 256, 6, 6, 130, 3, 3, pre=(1, 1), post=(1, 1))
    x = np.full(cfg.x_dims, -128, dtype=np.int8)
    w = np.full(cfg.w_dims, -128, dtype=np.int8)
    got, ref = _run_both(ic, cfg, algo=1, x=x, w=w, b=None)
    assert ref[0, 0, 2, 2] == 256 * 9 * 16384
    _assert_equal(got, ref, "all -128")


def test_group_sum_reaches_two_to_24(ic):
    """One group of 1024 products of 2^14 sums to exactly 2^24; mixed signs
    and magnitudes near the extremes around it."""
    cfg = synth.ConvConfig("g24", 1, 2048, 3, 3, 16, 1, 1)
    x = np.full(cfg.x_dims, -128, dtype=np.int8)
    w = np.full(cfg.w_dims, -128, dtype=np.int8)
    w[1, 1024:] = 127      # second half of the reduction flips sign
    w[2, ::2] = 127        # alternating
    w[3, :] = -127
    x[0, ::3, 1, 1] = 127
    got, ref = _run_both(ic, cfg, algo=1, x=x, w=w, b=None)
    assert ref[0, 0, 0, 0] == 2048 * 16384
    _assert_equal(got, ref, "2^24 groups")


def test_random_extremes_full_reduction(ic):
    cfg = synth.ConvConfig("ext", 2, 512, 7, 7, 64, 3, 3, pre=(1, 1), post=(1, 1), extremes=0.5, seed=31)
    got, ref = _run_both(ic, cfg, algo=1)
    _assert_equal(got, ref, "random extremes")


# ------------------------------------------------------------------ host buffers
@pytest.mark.parametrize("name,batch,pinned", [("c2_s2_nhwc", None, True), ("c4_1x1_bias_relu", None, True),
                                               ("c5_7x1_dilated_conv", 3, True), ("p4_shape", None, False),
                                               ("c3_3x3_large", 5, False)])
def test_host_buffer_pipeline(ic, name, batch, pinned):
    """conv_fprop_host: tensors in host memory, batch pipelined in chunks."""
    import dataclasses
    cfg = synth.CONFIGS[name] if batch is None else dataclasses.replace(synth.CONFIGS[name], N=batch)
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))

    def host(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.pin_memory() if pinned else t

    xh, wh = host(xf), host(wf)
    bh = host(b) if b is not None else None
    yh = torch.full((ysz,), -3, dtype=torch.int32)
    yh = yh.pin_memory() if pinned else yh
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    yd = ic.TensorDesc.make(ic.CONV_INT32, cfg.y_dims, ystr, ysz * 4)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
    need = ic.host_buffer_size(xd, wd, yd, p)
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    st = ic.conv_fprop_host_raw(xd, xh.data_ptr(), wd, wh.data_ptr(), yd, yh.data_ptr(),
                                bh.data_ptr() if bh is not None else 0, p, buf.data_ptr(), need, s.cuda_stream)
    assert st == 0, ic.STATUS.get(st)
    s.synchronize()
    assert ic.device_status() == 0
    got = synth.gather_logical(yh.numpy(), cfg.y_dims, ystr)
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, b, cfg.relu)
    _assert_equal(got, ref, f"host pipeline {name}")


def test_host_buffer_pipeline_int8_output(ic):
    """conv_fprop_host with int8 output: chunk sizes and copies by the 1-byte
    element (5 images of the 3x3 workload at full spatial size)."""
    import dataclasses
    cfg = dataclasses.replace(synth.CONFIGS["c3_3x3_large"], N=5)
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))
    xh, wh = torch.from_numpy(xf).pin_memory(), torch.from_numpy(wf).pin_memory()
    yh = torch.full((ysz + 64,), 0x5A, dtype=torch.int8).pin_memory()
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    yd = ic.TensorDesc.make(ic.CONV_INT8, cfg.y_dims, ystr, ysz)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu, out_shift=9)
    need = ic.host_buffer_size(xd, wd, yd, p)
    buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    st = ic.conv_fprop_host_raw(xd, xh.data_ptr(), wd, wh.data_ptr(), yd, yh.data_ptr(), 0, p, buf.data_ptr(),
                                need, s.cuda_stream)
    assert st == 0, ic.STATUS.get(st)
    s.synchronize()
    assert ic.device_status() == 0
    yn = yh.numpy()
    assert np.all(yn[ysz:] == 0x5A), "write past the output"
    got = synth.gather_logical(yn[:ysz], cfg.y_dims, ystr)
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, b, cfg.relu, out_int8=True, out_shift=9)
    _assert_equal(got, ref, "host pipeline int8 output")


# ------------------------------------------------------------------ edge cases and status
def test_empty_batch_is_a_no_op(ic):
    x = torch.zeros((0, 64, 8, 8), dtype=torch.int8, device="cuda").to(memory_format=torch.channels_last)
    w = torch.zeros((16, 64, 3, 3), dtype=torch.int8, device="cuda").to(memory_format=torch.channels_last)
    y = ic.conv_fprop(x, w, padding=(1, 1))
    assert tuple(y.shape) == (0, 16, 8, 8)


def test_single_pixel_output(ic):
    cfg = synth.ConvConfig("one_pixel", 1, 64, 3, 3, 8, 3, 3, seed=41)
    for algo in ALGOS:
        got, ref = _run_both(ic, cfg, algo=algo)
        _assert_equal(got, ref, f"1x1 output algo {algo}")


def test_timeout_is_reported_and_cleared(ic):
    assert ic.device_status() == 0
    assert ic.selftest_wait_timeout(2000) == 0
    assert ic.device_status() == ic.STATUS_CODE["CONV_ERR_DEVICE_TIMEOUT"]
    assert ic.device_status() == 0
    # the context still works afterwards
    got, ref = _run_both(ic, synth.CONFIGS["c1_tiny_nchw"])
    _assert_equal(got, ref, "after timeout")


def test_workspace_too_small_is_refused(ic):
    cfg = synth.CONFIGS["c2_s2_nhwc"]
    xd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.x_dims, cfg.x_layout)
    wd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.w_dims, cfg.w_layout)
    yd = ic.TensorDesc.packed(ic.CONV_INT32, cfg.y_dims, cfg.y_layout)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride)
    need = ic.workspace_size(xd, wd, yd, p)
    x = torch.zeros(xd.capacity_bytes, dtype=torch.int8, device="cuda")
    w = torch.zeros(wd.capacity_bytes, dtype=torch.int8, device="cuda")
    y = torch.zeros(yd.capacity_bytes // 4, dtype=torch.int32, device="cuda")
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert ic.conv_fprop_raw(xd, x.data_ptr(), wd, w.data_ptr(), yd, y.data_ptr(), 0, p, ws.data_ptr(),
                             need - 256, s) == ic.STATUS_CODE["CONV_ERR_WORKSPACE"]
    assert ic.conv_fprop_raw(xd, x.data_ptr(), wd, w.data_ptr(), yd, y.data_ptr(), 0, p, ws.data_ptr(),
                             need, s) == 0
    torch.cuda.synchronize()
