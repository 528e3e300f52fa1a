"""conv_fprop_static_workspace: the entry point for callers that cannot
allocate device memory (a plugin whose host framework hands it no
workspace, a latency-critical loop that must not call cudaMalloc).  Its
scratch is the library's own static device array.

Checked through the C ABI against conv_fprop with a caller workspace and
against the CPU oracle, bit for bit (tolerance 0, as everywhere for this
integer path), on two calls in a row: the second call runs with the array
still holding the first call's scratch.  A repeated call is also checked to
leave the device's free memory and torch's allocations unchanged.  Runs last
in the suite (file name), and also alone in a fresh process (the first call
on the device looks up the array's address)."""
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


def _device_case(ic, cfg):
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))
    dev = dict(x=torch.from_numpy(xf).cuda(), w=torch.from_numpy(wf).cuda(),
               b=torch.from_numpy(b).cuda() if b is not None else None)
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    yd = ic.TensorDesc.make(ic.CONV_INT32, cfg.y_dims, ystr, ysz * 4)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
    return dev, xd, wd, yd, p, ysz


def _oracle(cfg):
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride, cfg.dilation,
                            cfg.mode, b, cfg.relu)
    # logical [N,K,P,Q] -> the packed output layout the calls write
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    flat = np.empty(int(np.prod(cfg.y_dims)), dtype=np.int32)
    np.lib.stride_tricks.as_strided(flat, shape=cfg.y_dims, strides=tuple(4 * v for v in ystr))[...] = ref
    return flat


def _both(ic, cfg):
    dev, xd, wd, yd, p, ysz = _device_case(ic, cfg)
    s = torch.cuda.current_stream().cuda_stream
    bptr = dev["b"].data_ptr() if dev["b"] is not None else 0
    need = ic.workspace_size(xd, wd, yd, p)
    assert 0 < need <= 32 << 20
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    y_ref = torch.full((ysz,), -7, dtype=torch.int32, device="cuda")
    y_new = torch.full((ysz,), -9, dtype=torch.int32, device="cuda")
    assert ic.conv_fprop_raw(xd, dev["x"].data_ptr(), wd, dev["w"].data_ptr(), yd, y_ref.data_ptr(), bptr, p,
                             ws.data_ptr(), need, s) == 0
    assert ic.conv_fprop_static_workspace_raw(xd, dev["x"].data_ptr(), wd, dev["w"].data_ptr(), yd,
                                              y_new.data_ptr(), bptr, p, s) == 0
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    return y_ref.cpu().numpy(), y_new.cpu().numpy()


def test_static_workspace_matches_conv_fprop_twice(ic):
    import dataclasses
    first = synth.CONFIGS["c2_s2_nhwc"]
    # NCHW image: this call also uses the array for the channels-last copy
    second = dataclasses.replace(synth.CONFIGS["c5_7x1_dilated_conv"], N=2)
    for cfg in (first, second):
        ref, new = _both(ic, cfg)
        assert np.array_equal(ref, new), f"{cfg.name}: {int(np.sum(ref != new))} outputs differ from conv_fprop"
        truth = _oracle(cfg)
        assert np.array_equal(truth, new), f"{cfg.name}: {int(np.sum(truth != new))} outputs differ from the oracle"


def test_static_workspace_call_allocates_nothing(ic):
    cfg = synth.CONFIGS["c2_s2_nhwc"]
    dev, xd, wd, yd, p, ysz = _device_case(ic, cfg)
    s = torch.cuda.current_stream().cuda_stream
    y = torch.empty(ysz, dtype=torch.int32, device="cuda")

    def call():
        assert ic.conv_fprop_static_workspace_raw(xd, dev["x"].data_ptr(), wd, dev["w"].data_ptr(), yd,
                                                  y.data_ptr(), 0, p, s) == 0
        torch.cuda.synchronize()

    call()  # first call on the device: looks up the array's address, loads the kernels
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(3):
        call()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert ic.device_status() == 0
    assert np.array_equal(y.cpu().numpy(), _oracle(cfg))


def test_static_workspace_refuses_calls_beyond_its_size(ic):
    # an NCHW image whose channels-last copy alone exceeds 32 MiB
    cfg = synth.ConvConfig("too_big", 4, 512, 128, 130, 64, 3, 3, pre=(1, 1), post=(1, 1),
                           x_layout="NCHW", w_layout="KCRS", y_layout="NCHW")
    xd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.x_dims, cfg.x_layout)
    wd = ic.TensorDesc.packed(ic.CONV_INT8, cfg.w_dims, cfg.w_layout)
    yd = ic.TensorDesc.packed(ic.CONV_INT32, cfg.y_dims, cfg.y_layout)
    p = ic.Params.make(cfg.pre, cfg.post)
    assert ic.workspace_size(xd, wd, yd, p) > 32 << 20
    st = ic.conv_fprop_static_workspace_raw(xd, 0x10000000, wd, 0x20000000, yd, 0x40000000, 0, p, 0)
    assert ic.STATUS[st] == "CONV_ERR_STATIC_WORKSPACE_LIMIT"
