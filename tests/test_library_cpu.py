"""Host-side checks of libint8conv.so that need no GPU: the library loads and
exports every entry point of include/int8conv.h, the stride calculator, the
output-size rule and every rejection rule of the validator (including the two
descriptor sets of the forum thread "INT8 convolution using cuDNN Python
Frontend"), the planner's choices and workspace sizes, and the argument checks
conv_fprop makes before it touches a device."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ic():
    import __graft_entry__
    __graft_entry__.build_library()
    import int8_conv2d_fprop_gb300 as m
    m.lib()
    return m


def _descs(ic, cfg, y_layout=None):
    xd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.x_dims, cfg.x_layout)
    wd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.w_dims, cfg.w_layout)
    yd = ic.TensorDesc.packed(ic.CONV_INT32, cfg.y_dims, y_layout or cfg.y_layout)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
    return xd, wd, yd, p


def test_exports_every_declared_entry_point(ic):
    header = open(os.path.join(ROOT, "include", "int8conv.h")).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(conv_[a-z_0-9]+)\s*\(", header, re.M))
    assert declared == set(ic.EXPORTED_SYMBOLS)
    out = subprocess.run(["nm", "-D", "--defined-only", ic._LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (conv_[a-z_0-9]+)$", out, re.M))
    assert declared <= exported
    for name in declared:
        assert hasattr(ic.lib(), name)


def test_status_strings_cover_every_code(ic):
    for code, name in ic.STATUS.items():
        assert ic.status_string(code).startswith(name)
    assert ic.lib().conv_library_version() >= 100


def test_params_defaults_and_symmetric_padding(ic):
    p = ic.Params()
    ic.lib().conv_params_init(ctypes.byref(p))
    assert tuple(p.stride) == (1, 1) and tuple(p.dilation) == (1, 1)
    assert tuple(p.pre_padding) == (0, 0) and tuple(p.post_padding) == (0, 0)
    assert p.mode == ic.CROSS_CORRELATION and p.compute_dtype == ic.CONV_INT32 and p.algo == 0
    q = ic.Params.make(padding=(3, 2))
    assert tuple(q.pre_padding) == (3, 2) and tuple(q.post_padding) == (3, 2)


@pytest.mark.parametrize("layout", ["NCHW", "NHWC", "KCRS", "KRSC"])
def test_stride_calculator_matches_packed_layouts(ic, layout):
    dims = (2, 3, 5, 7)
    d = ic.TensorDesc.packed(ic.CONV_INT8, dims, layout)
    assert d.strides_t == synth.packed_strides(dims, layout)
    assert d.capacity_bytes == 2 * 3 * 5 * 7
    d32 = ic.TensorDesc.packed(ic.CONV_INT32, dims, layout)
    assert d32.capacity_bytes == 4 * 2 * 3 * 5 * 7
    with pytest.raises(ic.ConvError):
        ic.TensorDesc.packed(ic.CONV_INT8, dims, "NWHC")


@pytest.mark.parametrize("name", sorted(synth.CONFIGS))
def test_output_dims_and_validation_of_workloads(ic, name):
    cfg = synth.CONFIGS[name]
    xd, wd, yd, p = _descs(ic, cfg)
    assert ic.output_dims(xd, wd, p) == cfg.y_dims
    assert ic.output_dims(xd, wd, p) == oracle.out_dims(cfg.x_dims, cfg.w_dims, cfg.pre, cfg.post,
                                                        cfg.stride, cfg.dilation)
    assert ic.validate(xd, wd, yd, p, cfg.K if cfg.bias else 0) == 0


def test_forum_descriptors_are_both_valid(ic):
    """Both stride sets of the forum thread describe the same bytes (C = 1)."""
    p = ic.Params.make(padding=(0, 0))
    for xs, ws in (((25, 1, 5, 1), (9, 1, 3, 1)), ((25, 25, 5, 1), (9, 9, 3, 1))):
        xd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 5, 5), xs, 25)
        wd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 3, 3), ws, 9)
        yd = ic.TensorDesc.make(ic.CONV_INT32, (1, 1, 3, 3), (9, 9, 3, 1), 36)
        assert ic.validate(xd, wd, yd, p) == 0


def test_forum_failure_output_typed_int8_is_rejected(ic):
    """The forum thread's output was left to default to the int8 I/O type; an
    output descriptor that is not INT32 is refused."""
    p = ic.Params.make()
    xd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 5, 5), (25, 25, 5, 1), 25)
    wd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 3, 3), (9, 9, 3, 1), 9)
    yd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 3, 3), (9, 9, 3, 1), 36)
    assert ic.validate(xd, wd, yd, p) == ic.STATUS_CODE["CONV_ERR_DTYPE"]
    wd32 = ic.TensorDesc.make(ic.CONV_INT32, (1, 1, 3, 3), (9, 9, 3, 1), 36)
    yd32 = ic.TensorDesc.make(ic.CONV_INT32, (1, 1, 3, 3), (9, 9, 3, 1), 36)
    assert ic.validate(xd, wd32, yd32, p) == ic.STATUS_CODE["CONV_ERR_DTYPE"]


def _base(ic):
    cfg = synth.CONFIGS["c2_s2_nhwc"]
    return cfg, _descs(ic, cfg)


def _code(ic, name):
    return ic.STATUS_CODE[name]


def test_validator_rejections(ic):
    cfg, (xd, wd, yd, p) = _base(ic)
    assert ic.validate(xd, wd, yd, p) == 0

    def mod(desc, **kw):
        d = ic.TensorDesc.make(desc.dtype, desc.dims_t, desc.strides_t, desc.capacity_bytes)
        for k, v in kw.items():
            if k in ("dims", "strides"):
                for i in range(4):
                    getattr(d, k)[i] = v[i]
            else:
                setattr(d, k, v)
        return d

    # aliasing strides (two dims map onto the same bytes)
    bad = mod(xd, strides=(xd.strides[0], 1, xd.strides[2], 32))
    assert ic.validate(bad, wd, yd, p) == _code(ic, "CONV_ERR_BAD_STRIDES")
    # zero and negative strides of a dim larger than one
    assert ic.validate(mod(xd, strides=(xd.strides[0], 1, 0, 64)), wd, yd, p) == _code(ic, "CONV_ERR_BAD_STRIDES")
    assert ic.validate(mod(xd, strides=(xd.strides[0], 1, -3584, 64)), wd, yd, p) == _code(ic, "CONV_ERR_BAD_STRIDES")
    # buffer smaller than the extent
    assert ic.validate(xd, wd, mod(yd, capacity_bytes=yd.capacity_bytes - 4), p) == _code(ic, "CONV_ERR_BUFFER_TOO_SMALL")
    assert ic.validate(mod(xd, capacity_bytes=xd.capacity_bytes - 1), wd, yd, p) == _code(ic, "CONV_ERR_BUFFER_TOO_SMALL")
    # rank and dtype
    assert ic.validate(mod(xd, rank=3), wd, yd, p) == _code(ic, "CONV_ERR_RANK")
    assert ic.validate(mod(xd, dtype=ic.CONV_INT32), wd, yd, p) == _code(ic, "CONV_ERR_DTYPE")
    # channel mismatch between image and filter
    wbad = ic.TensorDesc.packed(ic.CONV_INT8, (64, 32, 3, 3), "KRSC")
    assert ic.validate(xd, wbad, yd, p) == _code(ic, "CONV_ERR_SHAPE_MISMATCH")
    # output dims that are not the computed P, Q
    ybad = ic.TensorDesc.packed(ic.CONV_INT32, (8, 64, 27, 28), "NHWC")
    assert ic.validate(xd, wd, ybad, p) == _code(ic, "CONV_ERR_SHAPE_MISMATCH")
    ybad = ic.TensorDesc.packed(ic.CONV_INT32, (8, 32, 28, 28), "NHWC")
    assert ic.validate(xd, wd, ybad, p) == _code(ic, "CONV_ERR_SHAPE_MISMATCH")
    # parameters
    for kw in (dict(stride=(0, 1)), dict(dilation=(1, 0)), dict(pre_padding=(-1, 0), post_padding=(1, 1))):
        args = dict(pre_padding=(1, 1), post_padding=(1, 1), stride=(2, 2))
        args.update(kw)
        assert ic.validate(xd, wd, yd, ic.Params.make(**args)) == _code(ic, "CONV_ERR_BAD_PARAM")
    pm = ic.Params.make((1, 1), (1, 1), (2, 2), mode=2)
    assert ic.validate(xd, wd, yd, pm) == _code(ic, "CONV_ERR_BAD_PARAM")
    pc = ic.Params.make((1, 1), (1, 1), (2, 2), compute_dtype=ic.CONV_INT8)
    assert ic.validate(xd, wd, yd, pc) == _code(ic, "CONV_ERR_UNSUPPORTED_COMPUTE")
    # bias requested but too short
    pb = ic.Params.make((1, 1), (1, 1), (2, 2), bias=True)
    assert ic.validate(xd, wd, yd, pb, 63) == _code(ic, "CONV_ERR_BUFFER_TOO_SMALL")
    assert ic.validate(xd, wd, yd, pb, 64) == 0
    # empty output (filter wider than the padded image)
    xs = ic.TensorDesc.packed(ic.CONV_INT8, (1, 4, 2, 2), "NHWC")
    ws = ic.TensorDesc.packed(ic.CONV_INT8, (4, 4, 3, 3), "KRSC")
    out = (ctypes.c_int64 * 4)()
    assert ic.lib().conv_fprop_output_dims(ctypes.byref(xs), ctypes.byref(ws), ctypes.byref(ic.Params.make()),
                                           out) == _code(ic, "CONV_ERR_BAD_PARAM")


def test_overflow_bound(ic):
    """C*R*S*2^14 must fit int32: 131071 taps pass, 131072 are refused."""
    p = ic.Params.make()
    for crs, ok in ((131071, True), (131072, False)):
        xd = ic.TensorDesc.packed(ic.CONV_INT8, (1, crs, 1, 1), "NHWC")
        wd = ic.TensorDesc.packed(ic.CONV_INT8, (1, crs, 1, 1), "KRSC")
        yd = ic.TensorDesc.packed(ic.CONV_INT32, (1, 1, 1, 1), "NHWC")
        st = ic.validate(xd, wd, yd, p)
        assert (st == 0) == ok
        if not ok:
            assert st == _code(ic, "CONV_ERR_OVERFLOW_RISK")
    assert oracle.worst_case_abs(131071, 1, 1) <= 2 ** 31 - 1 < oracle.worst_case_abs(131072, 1, 1)


def test_unit_dim_strides_are_ignored(ic):
    p = ic.Params.make()
    xd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 5, 5), (0, -7, 5, 1), 25)
    wd = ic.TensorDesc.make(ic.CONV_INT8, (1, 1, 3, 3), (123, 0, 3, 1), 9)
    yd = ic.TensorDesc.make(ic.CONV_INT32, (1, 1, 3, 3), (0, 0, 3, 1), 36)
    assert ic.validate(xd, wd, yd, p) == 0


def test_planner_choices_and_workspace(ic):
    algo = {}
    ws = {}
    kernels = {}
    for name, cfg in synth.CONFIGS.items():
        xd, wd, yd, p = _descs(ic, cfg)
        algo[name] = ic.plan(xd, wd, yd, p)
        ws[name] = ic.workspace_size(xd, wd, yd, p)
        kernels[name] = ic.kernel_count(xd, wd, yd, p)
    # kernels per call: one direct kernel; the convolution alone where the
    # 128- and 192-column kernels convert a channels-contiguous (KRSC)
    # filter themselves (C2, C4); filter repack + convolution otherwise (C3's
    # 256-column tiles, C5's KCRS filter; C5's NCHW image is read in place,
    # whole rows per k-step); no GPU here: one SM, so no call cuts its tiles
    assert kernels == {"c1_tiny_nchw": 1, "p4_shape": 1, "c2_s2_nhwc": 1, "c3_3x3_large": 2,
                       "c4_1x1_bias_relu": 1, "c5_7x1_dilated_conv": 2}
    # an empty batch launches nothing
    cfg = synth.CONFIGS["c3_3x3_large"]
    xd = ic.TensorDesc.make(ic.CONV_INT8, (0, 256, 56, 56), (56 * 56 * 256, 1, 56 * 256, 256), 0)
    yd = ic.TensorDesc.make(ic.CONV_INT32, (0, 256, 56, 56), (56 * 56 * 256, 1, 56 * 256, 256), 0)
    _, wd, _, p = _descs(ic, cfg)
    assert ic.kernel_count(xd, wd, yd, p) == 0
    assert algo["c1_tiny_nchw"] == ic.ALGO_DIRECT_DP4A
    assert algo["p4_shape"] == ic.ALGO_DIRECT_DP4A
    for name in ("c2_s2_nhwc", "c3_3x3_large", "c4_1x1_bias_relu", "c5_7x1_dilated_conv"):
        assert algo[name] == ic.ALGO_IMPLICIT_GEMM
    assert ws["c1_tiny_nchw"] == 0 and ws["p4_shape"] == 0
    # C3: 2 n-tiles x 36 k-steps x 16 KB of f16 filter blocks, no image copy
    assert ws["c3_3x3_large"] == 2 * 36 * 16384
    # C5 (K = 192: one 192-column tile, 14 k-steps of 192 rows x 128 bytes)
    # reads its NCHW image in place: the workspace holds the filter only
    assert ws["c5_7x1_dilated_conv"] == 14 * 192 * 128
    # forced algorithms are honoured
    xd, wd, yd, p = _descs(ic, synth.CONFIGS["c2_s2_nhwc"])
    for a in (ic.ALGO_DIRECT_GENERIC, ic.ALGO_DIRECT_DP4A, ic.ALGO_IMPLICIT_GEMM,
              ic.ALGO_IMPLICIT_GEMM_GLOBAL_LOADS):
        p.algo = a
        assert ic.plan(xd, wd, yd, p) == a
        tensor_core = a in (ic.ALGO_IMPLICIT_GEMM, ic.ALGO_IMPLICIT_GEMM_GLOBAL_LOADS)
        assert (ic.workspace_size(xd, wd, yd, p) > 0) == tensor_core
    p.algo = 5
    assert ic.validate(xd, wd, yd, p) == _code(ic, "CONV_ERR_BAD_PARAM")


def test_tile_shape_query(ic):
    """conv_fprop_tile_shape: pixels and channels per tile, tiles and work
    units of the implicit GEMM; zeros for the direct kernels.  Without a GPU
    the planner assumes one SM, so no call cuts its tiles."""
    shapes = {name: ic.tile_shape(*_descs(ic, cfg)) for name, cfg in synth.CONFIGS.items()}
    assert shapes["c1_tiny_nchw"] == (0, 0, 0, 0) and shapes["p4_shape"] == (0, 0, 0, 0)
    assert shapes["c2_s2_nhwc"] == (128, 128, 49, 49)
    assert shapes["c3_3x3_large"] == (128, 256, 784, 784)
    assert shapes["c4_1x1_bias_relu"] == (128, 128, 392, 392)
    assert shapes["c5_7x1_dilated_conv"] == (128, 192, 672, 672)
    xd, wd, yd, p = _descs(ic, synth.CONFIGS["c4_1x1_bias_relu"])
    st = ic.lib().conv_fprop_tile_shape(ctypes.byref(xd), ctypes.byref(wd), ctypes.byref(yd), ctypes.byref(p), None)
    assert st == _code(ic, "CONV_ERR_NULL_PTR")


def test_wgrad_fold_rule(ic):
    """The weight gradient folds T = min(64 / N, Q, 8) columns of dY into the
    channels for a batch N <= 32: its workspace is the folded filter blocks
    (K rows per tile x P * ceil(Q / T) taps x 128 bytes) plus the image copy
    X'' (C images x H rows x U columns x ceil(T*N / 16)*16 channels, U =
    T*stride_w*(ceil(Q/T) - 1) + dilation_w*(S - 1) + 1); larger batches
    keep one tap per k-step (their image copied channels-last with
    ceil(N / 16)*16 channels).  One SM here: no split partial sums."""
    def d(dtype, dims, layout):
        return ic.TensorDesc.packed(dtype, dims, layout)

    def ws(N, C, H, W, K):
        x = d(ic.CONV_INT8, (N, C, H, W), "NHWC")
        dy = d(ic.CONV_INT8, (N, K, H, W), "NHWC")
        dw = d(ic.CONV_INT32, (K, C, 3, 3), "KRSC")
        return ic.wgrad_workspace_size(x, dy, dw, ic.Params.make(padding=(1, 1)))

    # the 3x3 workload: T = 2, 28 folded columns, 256-row tiles, U = 57
    assert ws(32, 256, 56, 56, 256) == 56 * 28 * 256 * 128 + 256 * 56 * 57 * 64
    # batch 33 and 40: unfolded, 14 x 14 taps of one 128-row tile
    for n in (33, 40):
        c16 = (n + 15) // 16 * 16
        assert ws(n, 64, 14, 14, 32) == 14 * 14 * 128 * 128 + 64 * 14 * 14 * c16
    # batch 5: T = 8 (not 12), two folded columns, 48 channels
    assert ws(5, 64, 14, 14, 32) == 14 * 2 * 128 * 128 + 64 * 14 * 11 * 48


@pytest.mark.parametrize("W,pre_w,dil_w,S,K,stride_w,in_place", [
    (96, 0, 1, 1, 192, 1, True),     # the 7x1 workload's rows: two output rows per tile
    (64, 0, 1, 1, 128, 1, True),
    (32, 4, 4, 3, 96, 1, True),      # tap offsets 0, 4, 8 around pre-padding 4
    (16, 0, 1, 1, 128, 1, True),     # 16-byte rows, eight per tile
    (20, 0, 1, 1, 128, 1, False),    # rows not a multiple of 16 bytes
    (208, 0, 1, 1, 128, 1, False),   # rows longer than 192 bytes
    (112, 0, 1, 1, 128, 1, False),   # a tile's two rows exceed the 192-byte slot row
    (96, 1, 1, 3, 128, 1, False),    # tap offsets not multiples of 4
    (96, 0, 2, 3, 128, 1, False),    # dilation 2 along W with three taps
    (96, 0, 1, 1, 256, 1, False),    # 256-column tiles keep the channels-last copy
    (96, 0, 1, 1, 128, 2, False),    # stride 2 along W
])
def test_nchw_rows_planner_rules(ic, W, pre_w, dil_w, S, K, stride_w, in_place):
    """An NCHW image is read in place (no channels-last copy: two kernels,
    the workspace holds only the filter blocks) exactly when its rows are a
    multiple of 16 bytes and at most 192, the rows of one 128-pixel tile fit
    192 bytes per channel, the stride along W is 1, Q and every tap offset
    s*dil_w - pre_w are multiples of 4, and the tile has at most 192
    columns; otherwise the image is copied to channels-last first."""
    N, C, H = 2, 64, 10
    Q = (W + 2 * pre_w - dil_w * (S - 1) - 1) // stride_w + 1
    xd = ic.TensorDesc.packed(ic.CONV_INT8, (N, C, H, W), "NCHW")
    wd = ic.TensorDesc.packed(ic.CONV_INT8, (K, C, 1, S), "KCRS")
    yd = ic.TensorDesc.packed(ic.CONV_INT32, (N, K, H, Q), "NHWC")
    p = ic.Params.make((0, pre_w), (0, pre_w), (1, stride_w), (1, dil_w))
    n_tile = 128 if K <= 128 else (192 if K <= 192 else 256)
    filt = S * n_tile * 128  # S k-steps (one channel step) of n_tile rows x 64 f16
    copy = (N * H * W * 64 + 255) // 256 * 256
    # filter repack, unless a 128- or 192-column kernel over a channels-last
    # image (here: the copy) converts the filter itself, which it does when
    # the filter's channels are contiguous (KCRS with a 1x1 tap); image copy
    # unless read in place; the convolution
    self_filter = not in_place and n_tile <= 192 and S == 1
    assert ic.kernel_count(xd, wd, yd, p) == (0 if self_filter else 1) + (0 if in_place else 1) + 1
    assert ic.workspace_size(xd, wd, yd, p) == filt + (0 if in_place else copy)
    # gathering with global loads always takes the copy
    pg = ic.Params.make((0, pre_w), (0, pre_w), (1, stride_w), (1, dil_w), algo=ic.ALGO_IMPLICIT_GEMM_GLOBAL_LOADS)
    assert ic.workspace_size(xd, wd, yd, pg) == filt + copy


def test_host_buffer_size_covers_chunks(ic):
    """The host-pipeline device buffer holds the filter, the workspace and two
    image and two output chunks (a quarter of the batch each for C3)."""
    cfg = synth.CONFIGS["c3_3x3_large"]
    xd, wd, yd, p = _descs(ic, cfg)
    need = ic.host_buffer_size(xd, wd, yd, p)
    ws = ic.workspace_size(xd, wd, yd, p)
    x_chunk = 8 * 256 * 56 * 56
    y_chunk = 8 * 256 * 56 * 56 * 4
    assert need >= cfg.K * cfg.C * 9 + ws + 2 * x_chunk + 2 * y_chunk
    assert need < cfg.K * cfg.C * 9 + ws + 2 * x_chunk + 2 * y_chunk + 8 * 256


def test_int8_output_validation(ic):
    """INT8 output is an epilogue option: the output descriptor must be INT8
    exactly when CONV_EPILOGUE_INT8_OUT is set, with 0 <= out_shift <= 31;
    out_shift without the flag and a nonzero reserved word are refused."""
    cfg = synth.CONFIGS["c2_s2_nhwc"]
    xd, wd, yd32, p32 = _descs(ic, cfg)
    yd8 = ic.TensorDesc.packed(ic.CONV_INT8, cfg.y_dims, cfg.y_layout)
    assert yd8.capacity_bytes * 4 == yd32.capacity_bytes
    for s in (0, 1, 7, 31):
        p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, out_shift=s)
        assert p.epilogue & ic.EPILOGUE_INT8_OUT
        assert ic.validate(xd, wd, yd8, p) == 0
        # the flag with an int32 output descriptor, and int8 without the flag
        assert ic.validate(xd, wd, yd32, p) == _code(ic, "CONV_ERR_DTYPE")
    assert ic.validate(xd, wd, yd8, ic.Params.make(cfg.pre, cfg.post, cfg.stride)) == _code(ic, "CONV_ERR_DTYPE")
    for s in (-1, 32, 1000):
        p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, out_shift=s)
        assert ic.validate(xd, wd, yd8, p) == _code(ic, "CONV_ERR_BAD_PARAM")
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride)
    p.out_shift = 3
    assert ic.validate(xd, wd, yd32, p) == _code(ic, "CONV_ERR_BAD_PARAM")
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, out_shift=3)
    p.reserved = 1
    assert ic.validate(xd, wd, yd8, p) == _code(ic, "CONV_ERR_BAD_PARAM")
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, out_shift=3)
    small = ic.TensorDesc.make(ic.CONV_INT8, yd8.dims_t, yd8.strides_t, yd8.capacity_bytes - 1)
    assert ic.validate(xd, wd, small, p) == _code(ic, "CONV_ERR_BUFFER_TOO_SMALL")
    # the host pipeline sizes its output chunks by the output element size
    c3 = synth.CONFIGS["c3_3x3_large"]
    x3, w3, y3, p3 = _descs(ic, c3)
    y3_8 = ic.TensorDesc.packed(ic.CONV_INT8, c3.y_dims, c3.y_layout)
    p3_8 = ic.Params.make(c3.pre, c3.post, c3.stride, out_shift=8)
    need8 = ic.host_buffer_size(x3, w3, y3_8, p3_8)
    assert need8 < ic.host_buffer_size(x3, w3, y3, p3)
    # 25.7 MB of int8 output: three chunks of at least 8 MB, 11 images each
    per = 11
    x_chunk = per * c3.C * c3.H * c3.W
    y_chunk = per * c3.K * c3.P * c3.Q
    base = c3.K * c3.C * 9 + ic.workspace_size(x3, w3, y3_8, p3_8) + 2 * x_chunk + 2 * y_chunk
    assert base <= need8 < base + 8 * 256


def test_dp4a_refuses_long_reductions(ic):
    cfg = synth.CONFIGS["c3_3x3_large"]
    xd, wd, yd, p = _descs(ic, cfg)
    p.algo = ic.ALGO_DIRECT_DP4A
    with pytest.raises(ic.ConvError) as e:
        ic.plan(xd, wd, yd, p)
    assert e.value.name == "CONV_ERR_ALIGNMENT"


def test_call_checks_before_any_device_work(ic):
    cfg = synth.CONFIGS["c2_s2_nhwc"]
    xd, wd, yd, p = _descs(ic, cfg)
    code = ic.conv_fprop_raw(xd, 0, wd, 0x10000, yd, 0x20000000, 0, p, 0x40000000, 1 << 30, 0)
    assert code == _code(ic, "CONV_ERR_NULL_PTR")
    # output overlapping the image
    x = 0x10000000
    code = ic.conv_fprop_raw(xd, x, wd, 0x30000000, yd, x + 1024, 0, p, 0x40000000, 1 << 30, 0)
    assert code == _code(ic, "CONV_ERR_OVERLAP")
    # bias requested but no pointer
    pb = ic.Params.make(cfg.pre, cfg.post, cfg.stride, bias=True)
    code = ic.conv_fprop_raw(xd, x, wd, 0x30000000, yd, 0x50000000, 0, pb, 0x40000000, 1 << 30, 0)
    assert code == _code(ic, "CONV_ERR_NULL_PTR")
    # empty batch: nothing to do, nothing launched
    xe = ic.TensorDesc.packed(ic.CONV_INT8, (1, 64, 56, 56), "NHWC")
    xe.dims[0] = 0
    ye = ic.TensorDesc.packed(ic.CONV_INT32, (1, 64, 28, 28), "NHWC")
    ye.dims[0] = 0
    assert ic.conv_fprop_raw(xe, 0, wd, 0, ye, 0, 0, p, 0, 0, 0) == 0


def test_gradient_validation_and_routes(ic):
    """conv_dgrad / conv_wgrad take the forward call's descriptors and
    parameters: shapes, types, epilogue, algorithm and the int32 bound are
    checked; dgrad takes the tensor-core route (one forward convolution per
    residue class of the stride, each with its own workspace) up to 64
    classes, the CUDA-core kernel beyond that or when forced."""
    def d(dtype, dims, layout):
        return ic.TensorDesc.packed(dtype, dims, layout)

    x = d(ic.CONV_INT8, (2, 64, 14, 14), "NHWC")
    w = d(ic.CONV_INT8, (32, 64, 3, 3), "KRSC")
    dy = d(ic.CONV_INT8, (2, 32, 14, 14), "NHWC")
    dx = d(ic.CONV_INT32, (2, 64, 14, 14), "NHWC")
    dw = d(ic.CONV_INT32, (32, 64, 3, 3), "KRSC")
    p = ic.Params.make(padding=(1, 1))
    assert ic.dgrad_workspace_size(dy, w, dx, p) > 0          # tensor-core route
    # wgrad on the tensor cores: dY repacked as the filter of a forward
    # convolution, its batch of 2 folded with T = 8 of its 14 columns into 16
    # channels: one 128-channel tile (K = 32) x 14 x 2 taps x one channel
    # step of 64 f16 (128 bytes), then the image copy X'' of 64 images x 14
    # rows x 11 columns (8 * 1 * (2 - 1) + 1 * (3 - 1) + 1) x 16 channels
    assert ic.wgrad_workspace_size(x, dy, dw, p) == 14 * 2 * 128 * 128 + 64 * 14 * 11 * 16
    assert ic.wgrad_workspace_size(x, dy, dw, ic.Params.make(padding=(1, 1), algo=ic.ALGO_DIRECT_GENERIC)) == 0

    def code(fn, *a):
        try:
            fn(*a)
            return 0
        except ic.ConvError as e:
            return e.status

    S = ic.STATUS_CODE
    assert code(ic.dgrad_workspace_size, dy, w, d(ic.CONV_INT8, (2, 64, 14, 14), "NHWC"), p) == S["CONV_ERR_DTYPE"]
    assert code(ic.dgrad_workspace_size, dy, w, d(ic.CONV_INT32, (2, 64, 15, 14), "NHWC"), p) == \
        S["CONV_ERR_SHAPE_MISMATCH"]
    assert code(ic.wgrad_workspace_size, x, d(ic.CONV_INT8, (2, 31, 14, 14), "NHWC"), dw, p) == \
        S["CONV_ERR_SHAPE_MISMATCH"]
    pb = ic.Params.make(padding=(1, 1), relu=True)
    assert code(ic.dgrad_workspace_size, dy, w, dx, pb) == S["CONV_ERR_BAD_PARAM"]
    p8 = ic.Params.make(padding=(1, 1), out_shift=3)
    assert code(ic.wgrad_workspace_size, x, dy, dw, p8) == S["CONV_ERR_BAD_PARAM"]
    pa = ic.Params.make(padding=(1, 1), algo=ic.ALGO_DIRECT_DP4A)
    assert code(ic.dgrad_workspace_size, dy, w, dx, pa) == S["CONV_ERR_BAD_PARAM"]
    pg = ic.Params.make(padding=(1, 1), algo=ic.ALGO_IMPLICIT_GEMM)
    assert ic.wgrad_workspace_size(x, dy, dw, pg) > 0
    # stride 2: four residue classes on the tensor cores, each with its own
    # filter blocks (1 x 1, 1 x 2, 2 x 1 and 2 x 2 taps of the 3 x 3 filter,
    # one 128-channel tile, one channel step of 64 f16 per tap)
    dy2 = d(ic.CONV_INT8, (2, 32, 7, 7), "NHWC")
    p2 = ic.Params.make(pre_padding=(1, 1), post_padding=(0, 0), stride=(2, 2))
    assert ic.dgrad_workspace_size(dy2, w, dx, p2) == (1 + 2 + 2 + 4) * 128 * 128
    # padding wider than the filter's reach (3 > 2): one class, windows that
    # start inside dY
    dy3 = d(ic.CONV_INT8, (2, 32, 18, 18), "NHWC")
    p3 = ic.Params.make(padding=(3, 3))
    assert ic.dgrad_workspace_size(dy3, w, dx, p3) == 3 * 3 * 128 * 128
    # strides (9, 8): 72 classes, CUDA-core route, no workspace; forcing the
    # tensor cores is refused
    dy4 = d(ic.CONV_INT8, (2, 32, 2, 2), "NHWC")
    p4 = ic.Params.make(pre_padding=(1, 1), post_padding=(0, 0), stride=(9, 8))
    assert ic.dgrad_workspace_size(dy4, w, dx, p4) == 0
    p4g = ic.Params.make(pre_padding=(1, 1), post_padding=(0, 0), stride=(9, 8), algo=ic.ALGO_IMPLICIT_GEMM)
    assert code(ic.dgrad_workspace_size, dy4, w, dx, p4g) == S["CONV_ERR_ALIGNMENT"]
    # int32 bounds: dgrad sums K*R*S terms, wgrad N*P*Q terms
    wbig = d(ic.CONV_INT8, (14564, 64, 3, 3), "KRSC")    # 14564*9 = 131076 > 131071
    dybig = d(ic.CONV_INT8, (2, 14564, 14, 14), "NHWC")
    assert code(ic.dgrad_workspace_size, dybig, wbig, dx, p) == S["CONV_ERR_OVERFLOW_RISK"]
    xl = d(ic.CONV_INT8, (1, 8, 363, 363), "NHWC")      # 363*363 = 131769 > 131071 pixels
    dyl = d(ic.CONV_INT8, (1, 4, 363, 363), "NHWC")
    dwl = d(ic.CONV_INT32, (4, 8, 1, 1), "KRSC")
    assert code(ic.wgrad_workspace_size, xl, dyl, dwl, ic.Params.make()) == S["CONV_ERR_OVERFLOW_RISK"]
    xs = d(ic.CONV_INT8, (1, 8, 362, 362), "NHWC")      # 131044 pixels fit
    dys = d(ic.CONV_INT8, (1, 4, 362, 362), "NHWC")
    assert ic.wgrad_workspace_size(xs, dys, dwl, ic.Params.make()) >= 0


def _class_taps(rho, pre, stride, dil, taps):
    """Taps of one axis that reach the pixels h = rho (mod stride) of dX: the
    r with r*dil = rho + pre (mod stride), by direct enumeration."""
    return sum(1 for r in range(taps) if (r * dil - rho - pre) % stride == 0)


@pytest.mark.parametrize("stride,dil,pre,post,R,S", [
    ((2, 2), (1, 1), (1, 1), (0, 0), 3, 3),
    ((3, 2), (2, 3), (2, 1), (1, 2), 5, 4),
    ((2, 3), (2, 3), (0, 2), (1, 0), 3, 3),   # stride and dilation share a factor
    ((4, 4), (1, 1), (3, 3), (2, 3), 7, 7),
    ((2, 2), (1, 1), (0, 0), (0, 0), 1, 1),   # three of four classes untouched
    ((1, 1), (2, 1), (5, 0), (1, 2), 3, 3),   # padding wider than the reach (5 > 4)
])
@pytest.mark.parametrize("dy_layout", ["NHWC", "NCHW"])
def test_dgrad_residue_class_workspace(ic, stride, dil, pre, post, R, S, dy_layout):
    """The data gradient's workspace is the sum over the residue classes of
    the stride of each class's repacked filter: (taps of the class in H) x
    (taps in W) k-steps of 128 filter rows x 64 f16 channels (one tile of
    output channels, one channel step).  A dY that is not channels-last adds
    one channels-last copy (N x P x Q pixels x 48 channels, rounded up to 256
    bytes) that every class reads.  The tap counts come from enumerating the
    taps, not from the library's closed form."""
    def d(dtype, dims, layout):
        return ic.TensorDesc.packed(dtype, dims, layout)
    H, W = 23, 21
    P = (H + pre[0] + post[0] - dil[0] * (R - 1) - 1) // stride[0] + 1
    Q = (W + pre[1] + post[1] - dil[1] * (S - 1) - 1) // stride[1] + 1
    dy = d(ic.CONV_INT8, (2, 48, P, Q), dy_layout)
    w = d(ic.CONV_INT8, (48, 40, R, S), "KRSC")
    dx = d(ic.CONV_INT32, (2, 40, H, W), "NHWC")
    p = ic.Params.make(pre_padding=pre, post_padding=post, stride=stride, dilation=dil)
    want = 0
    tapped = 0
    for rh in range(stride[0]):
        for rw in range(stride[1]):
            th = _class_taps(rh, pre[0], stride[0], dil[0], R)
            tw = _class_taps(rw, pre[1], stride[1], dil[1], S)
            want += th * tw * 128 * 128  # zero taps: a zero-filled class, no workspace
            tapped += th * tw > 0
    if dy_layout == "NCHW" and tapped:
        want += (2 * P * Q * 48 + 255) // 256 * 256
    assert ic.dgrad_workspace_size(dy, w, dx, p) == want


def test_plan_cache_hits_and_shutdown(ic):
    """Repeated planning of one shape is served from the plan cache (no
    validation or planning again); conv_shutdown empties it; invalid calls
    are never cached."""
    cfg = synth.CONFIGS["c3_3x3_large"]
    xd, wd, yd, p = _descs(ic, cfg)
    ic.shutdown()
    s0 = ic.plan_cache_stats()
    a1 = ic.plan(xd, wd, yd, p)
    s1 = ic.plan_cache_stats()
    assert s1["plan_misses"] == s0["plan_misses"] + 1
    a2 = ic.plan(xd, wd, yd, p)
    w2 = ic.workspace_size(xd, wd, yd, p)
    s2 = ic.plan_cache_stats()
    assert a1 == a2 and w2 > 0
    assert s2["plan_hits"] == s1["plan_hits"] + 2 and s2["plan_misses"] == s1["plan_misses"]
    # another parameter set is another key
    p2 = ic.Params.make(cfg.pre, cfg.post, (2, 2), cfg.dilation, cfg.mode)
    xd2, wd2, _, _ = _descs(ic, cfg)
    yd2 = ic.TensorDesc.packed(ic.CONV_INT32, ic.output_dims(xd2, wd2, p2), cfg.y_layout)
    ic.plan(xd2, wd2, yd2, p2)
    assert ic.plan_cache_stats()["plan_misses"] == s2["plan_misses"] + 1
    # an invalid call (int8 output without the int8 epilogue) is refused every time
    bad = ic.TensorDesc.packed(ic.CONV_INT8, cfg.y_dims, cfg.y_layout)
    for _ in range(2):
        assert ic.validate(xd, wd, bad, p) != 0
        with pytest.raises(ic.ConvError):
            ic.plan(xd, wd, bad, p)
    ic.shutdown()
    s3 = ic.plan_cache_stats()
    ic.plan(xd, wd, yd, p)
    assert ic.plan_cache_stats()["plan_misses"] == s3["plan_misses"] + 1
