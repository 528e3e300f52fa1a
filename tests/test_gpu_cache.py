"""The plan and launch caches on the GPU: repeated calls of one shape on
different buffers (the cached tensor maps re-targeted to each call's
addresses), a change of pointer alignment (another cache key), and
conv_shutdown between calls -- every result compared with the CPU oracle
(tolerance 0)."""
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


@pytest.mark.parametrize("cfg", [
    synth.ConvConfig("cache_3x3_nt256", 2, 64, 20, 18, 256, 3, 3, pre=(1, 1), post=(1, 1), bias=True, seed=81),
    synth.ConvConfig("cache_1x1_tmem", 4, 128, 14, 14, 96, 1, 1, relu=True, seed=82),
    # NCHW image read in place (16-byte rows): the cached 4-D row map is re-targeted
    synth.ConvConfig("cache_nchw_rows", 2, 48, 16, 16, 150, 3, 1, stride=(2, 1), pre=(1, 0), post=(1, 0),
                     x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=83),
    # NCHW image copied to channels-last (20-byte rows): the map of the copy
    synth.ConvConfig("cache_nchw_packed", 2, 48, 16, 20, 150, 3, 1, stride=(2, 1), pre=(1, 0), post=(1, 0),
                     x_layout="NCHW", w_layout="KCRS", y_layout="NCHW", seed=84),
], ids=lambda c: c.name)
def test_cached_calls_on_other_buffers(ic, cfg):
    x, w, b = synth.make_inputs(cfg)
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride, cfg.dilation,
                            cfg.mode, b, cfg.relu)
    ystr = synth.packed_strides(cfg.y_dims, cfg.y_layout)
    ysz = int(np.prod(cfg.y_dims))
    xd = ic.TensorDesc.make(ic.CONV_INT8, cfg.x_dims, xs, xf.size)
    wd = ic.TensorDesc.make(ic.CONV_INT8, cfg.w_dims, ws, wf.size)
    yd = ic.TensorDesc.make(ic.CONV_INT32, cfg.y_dims, ystr, ysz * 4)
    p = ic.Params.make(cfg.pre, cfg.post, cfg.stride, cfg.dilation, cfg.mode, cfg.bias, cfg.relu)
    need = ic.workspace_size(xd, wd, yd, p)
    s = torch.cuda.current_stream().cuda_stream
    wt = torch.from_numpy(wf).cuda()
    bt = torch.from_numpy(b).cuda() if b is not None else None
    # three image / output / workspace sets, at 16-byte aligned offsets of
    # bigger buffers so that every call's addresses differ
    sets = []
    for k in range(3):
        xb = torch.zeros(xf.size + 256, dtype=torch.int8, device="cuda")
        xb[16 * (k + 1):16 * (k + 1) + xf.size].copy_(torch.from_numpy(xf))
        yb = torch.full((ysz + 64,), -1, dtype=torch.int32, device="cuda")
        wsb = torch.empty(need + 1024, dtype=torch.uint8, device="cuda")
        sets.append((xb, 16 * (k + 1), yb, 4 * (k + 1), wsb, 256 * k))
    ic.shutdown()
    before = ic.plan_cache_stats()
    for rep in range(2):
        for xb, xo, yb, yo, wsb, wo in sets:
            yb.fill_(-1)
            st = ic.conv_fprop_raw(xd, xb.data_ptr() + xo, wd, wt.data_ptr(), yd, yb.data_ptr() + 4 * yo,
                                   bt.data_ptr() if bt is not None else 0, p, wsb.data_ptr() + wo, need, s)
            assert st == 0, ic.STATUS.get(st)
            torch.cuda.synchronize()
            assert ic.device_status() == 0
            got = synth.gather_logical(yb[yo:yo + ysz].cpu().numpy(), cfg.y_dims, ystr)
            assert np.array_equal(got, ref), f"{cfg.name} rep {rep}: {int(np.sum(got != ref))} outputs differ"
    after = ic.plan_cache_stats()
    calls = 2 * len(sets)
    assert after["plan_misses"] - before["plan_misses"] == 1
    assert after["plan_hits"] - before["plan_hits"] == calls - 1
    assert after["launch_misses"] - before["launch_misses"] == 1
    assert after["launch_hits"] - before["launch_hits"] == calls - 1
    # an image pointer that is not 16-byte aligned is another key (and, for a
    # channels-last image or an NCHW image read in place, the path that
    # copies the image to channels-last first): still exact
    xb = torch.zeros(xf.size + 64, dtype=torch.int8, device="cuda")
    xb[8:8 + xf.size].copy_(torch.from_numpy(xf))
    # the aligned-pointer workspace size need not cover the image copy
    need2 = need + cfg.N * cfg.H * cfg.W * ((cfg.C + 15) // 16 * 16) + 4096
    wsb = torch.empty(need2 + 256, dtype=torch.uint8, device="cuda")
    yb = torch.full((ysz,), -1, dtype=torch.int32, device="cuda")
    st = ic.conv_fprop_raw(xd, xb.data_ptr() + 8, wd, wt.data_ptr(), yd, yb.data_ptr(),
                           bt.data_ptr() if bt is not None else 0, p, wsb.data_ptr(), need2, s)
    assert st == 0, ic.STATUS.get(st)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    got = synth.gather_logical(yb.cpu().numpy(), cfg.y_dims, ystr)
    assert np.array_equal(got, ref), f"{cfg.name} misaligned image"
