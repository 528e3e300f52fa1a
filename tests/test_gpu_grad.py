"""GPU parity of the gradients (conv_dgrad, conv_wgrad through the C ABI)
against the CPU oracle, element by element (integer results: tolerance 0).
Cases cover both dgrad routes (tensor cores, one forward convolution per
residue class of the stride; the CUDA-core kernel for more than 64 classes
or when forced), classes no tap reaches (zero-filled), classes whose windows
start inside dY (padding wider than the filter's reach), strides sharing a
factor with the dilation, both modes, NHWC and NCHW layouts and a ragged
tail."""
import dataclasses

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


@dataclasses.dataclass
class G:
    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    pre: tuple = (0, 0)
    post: tuple = (0, 0)
    stride: tuple = (1, 1)
    dil: tuple = (1, 1)
    mode: int = 0
    layout: str = "NHWC"
    algo: int = 0
    tensor: bool = False  # dgrad expected on the tensor-core route


CASES = [
    G("s1_3x3_pad1", 2, 64, 13, 11, 48, 3, 3, (1, 1), (1, 1), tensor=True),
    G("s1_5x3_dil_asym_conv", 2, 32, 12, 9, 40, 5, 3, (2, 1), (3, 2), dil=(2, 1), mode=1, tensor=True),
    G("s1_nchw_k200", 1, 24, 10, 10, 200, 3, 3, (0, 2), (2, 0), layout="NCHW", tensor=True),
    G("s1_generic_forced", 2, 16, 9, 8, 20, 3, 3, (1, 1), (1, 1), algo=3),
    G("s2_3x3", 2, 32, 15, 14, 24, 3, 3, (1, 1), (1, 0), stride=(2, 2), tensor=True),
    G("s21_dil_conv", 1, 8, 11, 12, 12, 3, 2, (2, 0), (0, 1), stride=(2, 1), dil=(1, 2), mode=1, tensor=True),
    G("pad_wider_than_reach", 2, 16, 6, 7, 8, 1, 1, (1, 2), (1, 0), tensor=True),
    G("s2_1x1_untouched_classes", 2, 64, 15, 16, 96, 1, 1, stride=(2, 2), tensor=True),
    G("s23_dil23_shared_factor", 1, 40, 17, 19, 72, 3, 3, (2, 2), (1, 2), stride=(2, 3), dil=(2, 3), tensor=True),
    G("s4_7x7_stem_nchw_conv", 2, 3, 32, 29, 64, 7, 7, (3, 3), (2, 3), stride=(4, 4), mode=1, layout="NCHW",
      tensor=True),
    G("s98_many_classes", 2, 16, 14, 14, 32, 3, 3, (1, 1), (0, 0), stride=(9, 8)),
    G("c3_shape_batch2", 2, 256, 56, 56, 256, 3, 3, (1, 1), (1, 1), tensor=True),
    G("c2_shape_s2_batch1", 1, 128, 56, 56, 256, 3, 3, (1, 1), (0, 0), stride=(2, 2), tensor=True),
    # strided classes launched together on 192- and 256-column tiles (the
    # classes' output channels are the forward image's C)
    G("s2_c160_group192", 2, 160, 21, 18, 48, 3, 3, (1, 1), (1, 1), stride=(2, 2), tensor=True),
    G("s2_c256_group256_conv", 1, 256, 17, 20, 40, 3, 2, (1, 0), (0, 1), stride=(2, 2), mode=1, tensor=True),
    # NCHW dY read in place (rows of 32 bytes, class windows at offsets that
    # are multiples of 4): one class; and a stride-2 1x1 filter whose one
    # tapped class writes every other dX pixel
    G("s1_nchw_rows_dy", 2, 48, 12, 32, 64, 3, 1, (1, 0), (1, 0), layout="NCHW", tensor=True),
    G("s2_1x1_nchw_rows_dy", 1, 64, 32, 64, 32, 1, 1, stride=(2, 2), layout="NCHW", tensor=True),
    # stride 2, 3x3, NCHW: some classes could read dY in place and some not;
    # all of them then read one shared channels-last copy
    G("s2_nchw_mixed_classes", 2, 32, 16, 32, 48, 3, 3, (1, 1), (1, 1), stride=(2, 2), layout="NCHW",
      tensor=True),
    # a batch of 70 (the weight gradient's channels: two channel steps, 80
    # bytes per pixel of its image copy, images (C = 80) in a full and a
    # ragged block of 64) and K = 48 rows of the repacked loss gradient
    G("batch70_c80_k48", 70, 80, 6, 7, 48, 3, 3, (1, 1), (1, 1), tensor=True),
    # a batch of 16 at stride 2: the weight gradient folds T = 4 of dY's 15
    # columns per k-step (four folded columns, the last one short), tap
    # dilation 8 along W over the image copy
    G("batch16_s2_fold4", 16, 24, 12, 30, 40, 3, 3, (1, 1), (1, 1), stride=(2, 2), tensor=True),
]


def _place(a, layout):
    f, s = synth.place(a, layout)
    return torch.as_strided(torch.from_numpy(np.ascontiguousarray(f)).cuda(), a.shape, s), f, s


def _setup(c):
    x = synth.int8_uniform(7000 + len(c.name), 1, (c.N, c.C, c.H, c.W))
    w = synth.int8_uniform(7000 + len(c.name), 2, (c.K, c.C, c.R, c.S))
    yd = oracle.out_dims(x.shape, w.shape, c.pre, c.post, c.stride, c.dil)
    dy = synth.int8_uniform(7000 + len(c.name), 3, yd)
    return x, w, dy


def _out(shape, layout):
    fmt = torch.channels_last if layout == "NHWC" else torch.contiguous_format
    return torch.full(shape, -999, dtype=torch.int32, device="cuda").to(memory_format=fmt)


@pytest.mark.parametrize("c", CASES, ids=lambda c: c.name)
def test_dgrad_matches_oracle(ic, c):
    x, w, dy = _setup(c)
    wl = "KRSC" if c.layout == "NHWC" else "KCRS"
    dyt, dyf, dys = _place(dy, c.layout)
    wt, wf, wss = _place(w, wl)
    dx = _out(x.shape, c.layout)
    kw = dict(pre_padding=c.pre, post_padding=c.post, stride=c.stride, dilation=c.dil, mode=c.mode, algo=c.algo)
    p = ic.Params.make(c.pre, c.post, c.stride, c.dil, c.mode, False, False, c.algo)
    route = ic.dgrad_workspace_size(ic.TensorDesc.from_tensor(dyt), ic.TensorDesc.from_tensor(wt),
                                    ic.TensorDesc.from_tensor(dx), p) > 0
    assert route == c.tensor
    ic.conv_dgrad(dyt, wt, out=dx, **kw)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    ref = oracle.conv_dgrad(dyf, dy.shape, dys, wf, w.shape, wss, x.shape, c.pre, c.post, c.stride, c.dil, c.mode)
    got = dx.cpu().numpy()
    assert np.array_equal(got, ref), f"{c.name}: {(got != ref).sum()} of {ref.size} dX elements differ"


@pytest.mark.parametrize("c", CASES, ids=lambda c: c.name)
def test_wgrad_matches_oracle(ic, c):
    x, w, dy = _setup(c)
    wl = "KRSC" if c.layout == "NHWC" else "KCRS"
    xt, xf, xs = _place(x, c.layout)
    dyt, dyf, dys = _place(dy, c.layout)
    dw = _out(w.shape, "NHWC" if wl == "KRSC" else "NCHW")  # KRSC is the NHWC order of [K,C,R,S]
    algo = 3 if c.algo == 3 else 0
    ic.conv_wgrad(xt, dyt, out=dw, pre_padding=c.pre, post_padding=c.post, stride=c.stride, dilation=c.dil,
                  mode=c.mode, algo=algo)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    ref = oracle.conv_wgrad(xf, x.shape, xs, dyf, dy.shape, dys, w.shape, c.pre, c.post, c.stride, c.dil, c.mode)
    got = dw.cpu().numpy()
    assert np.array_equal(got, ref), f"{c.name}: {(got != ref).sum()} of {ref.size} dW elements differ"


def test_dgrad_extremes_exceed_f32_integer_range(ic):
    """All -128 loss gradient and filter on the tensor-core route: interior dX
    sums are K*R*S*2^14 = 2304*16384 > 2^24, exact only with the grouped
    reduction."""
    c = G("ext", 1, 64, 12, 12, 256, 3, 3, (1, 1), (1, 1), tensor=True)
    dy = np.full((1, 256, 12, 12), -128, dtype=np.int8)
    w = np.full((256, 64, 3, 3), -128, dtype=np.int8)
    dyt, dyf, dys = _place(dy, "NHWC")
    wt, wf, wss = _place(w, "KRSC")
    dx = _out((1, 64, 12, 12), "NHWC")
    ic.conv_dgrad(dyt, wt, out=dx, padding=(1, 1))
    torch.cuda.synchronize()
    ref = oracle.conv_dgrad(dyf, dy.shape, dys, wf, w.shape, wss, (1, 64, 12, 12), (1, 1), (1, 1))
    assert int(ref.max()) == 256 * 9 * 16384
    assert np.array_equal(dx.cpu().numpy(), ref)


def test_wgrad_empty_batch_takes_null_inputs(ic):
    """An empty batch: dW is all zeros and neither input is read, so both
    input pointers may be null (only dW must be given)."""
    import ctypes
    x = ic.TensorDesc.make(ic.CONV_INT8, (0, 32, 9, 9), (9 * 9 * 32, 1, 9 * 32, 32), 0)
    dy = ic.TensorDesc.make(ic.CONV_INT8, (0, 48, 9, 9), (9 * 9 * 48, 1, 9 * 48, 48), 0)
    dwd = ic.TensorDesc.packed(ic.CONV_INT32, (48, 32, 3, 3), "NHWC")
    p = ic.Params.make(padding=(1, 1))
    out = torch.full((48 * 32 * 9,), 77, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = ic.lib().conv_wgrad(ctypes.byref(x), None, ctypes.byref(dy), None, ctypes.byref(dwd), out.data_ptr(),
                             ctypes.byref(p), None, 0, s)
    assert st == 0, ic.STATUS.get(st)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    assert int(out.abs().max()) == 0
    st = ic.lib().conv_wgrad(ctypes.byref(x), None, ctypes.byref(dy), None, ctypes.byref(dwd), None,
                             ctypes.byref(p), None, 0, s)
    assert ic.STATUS[st] == "CONV_ERR_NULL_PTR"


def _dgrad_case(ic, c):
    x, w, dy = _setup(c)
    wl = "KRSC" if c.layout == "NHWC" else "KCRS"
    dyt, dyf, dys = _place(dy, c.layout)
    wt, wf, wss = _place(w, wl)
    ref = oracle.conv_dgrad(dyf, dy.shape, dys, wf, w.shape, wss, x.shape, c.pre, c.post, c.stride, c.dil, c.mode)
    kw = dict(pre_padding=c.pre, post_padding=c.post, stride=c.stride, dilation=c.dil, mode=c.mode)
    return dyt, wt, x.shape, ref, kw


def test_dgrad_strided_repeated_calls_and_graph_replay(ic):
    """Strided data gradients called again and again with the same
    descriptors (the call's plan comes from the cache, its fork and join
    events are reused): fresh dY and dX buffers on every call, two shapes
    taking turns, then one call captured in a CUDA graph (the side streams
    fork from and join back into the capture) and replayed on new dY values.
    Every result is compared with the oracle."""
    cases = [c for c in CASES if c.name in ("s2_3x3", "s23_dil23_shared_factor")]
    assert len(cases) == 2
    for rep in range(3):
        for c in cases:
            dyt, wt, xshape, ref, kw = _dgrad_case(ic, c)
            dyt = dyt.clone(memory_format=torch.preserve_format)  # a fresh allocation each call
            dx = _out(xshape, c.layout)
            ic.conv_dgrad(dyt, wt, out=dx, **kw)
            torch.cuda.synchronize()
            assert ic.device_status() == 0
            got = dx.cpu().numpy()
            assert np.array_equal(got, ref), f"{c.name} call {rep}: {(got != ref).sum()} dX elements differ"
    c = cases[0]
    dyt, wt, xshape, ref, kw = _dgrad_case(ic, c)
    dx = _out(xshape, c.layout)
    p = ic.Params.make(c.pre, c.post, c.stride, c.dil, c.mode, False, False, 0)
    wsb = ic.dgrad_workspace_size(ic.TensorDesc.from_tensor(dyt), ic.TensorDesc.from_tensor(wt),
                                  ic.TensorDesc.from_tensor(dx), p)
    assert wsb > 0
    work = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        ic.conv_dgrad(dyt, wt, out=dx, workspace=work, stream=side, **kw)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        ic.conv_dgrad(dyt, wt, out=dx, workspace=work, stream=side, **kw)
    # new loss gradient values in the captured buffer, then replay
    dy2 = synth.int8_uniform(4242, 3, tuple(dyt.shape))
    dyt2, dyf2, dys2 = _place(dy2, c.layout)
    dyt.copy_(dyt2)
    dx.fill_(-5)
    graph.replay()
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    _, w, _ = _setup(c)
    wf, wss = synth.place(w, "KRSC" if c.layout == "NHWC" else "KCRS")
    ref2 = oracle.conv_dgrad(dyf2, dy2.shape, dys2, wf, w.shape, wss, xshape, c.pre, c.post, c.stride, c.dil,
                             c.mode)
    got = dx.cpu().numpy()
    assert np.array_equal(got, ref2), f"graph replay: {(got != ref2).sum()} dX elements differ"
