"""Every output of every workload at full size, in the launch configuration
the benchmark times: the benchmark's own DeviceWorkload (a step is one
conv_fprop call on resident inputs, with the cut last round and its
reduction kernel wherever the planner cuts one; the convolution-only timing
calls conv_fprop_pack_filter, then conv_fprop_prepacked), compared element
by element with the CPU oracle (tolerance 0).

The two large workloads take the oracle about 10 s (3x3, 118 G ops) and
3 s (7x1 dilated) on 16 host cores."""
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


@pytest.mark.parametrize("name", ["c1_tiny_nchw", "c2_s2_nhwc", "c3_3x3_large", "c4_1x1_bias_relu",
                                  "c5_7x1_dilated_conv"])
def test_every_output_at_full_size_as_benchmarked(ic, name):
    import bench
    cfg = synth.CONFIGS[name]
    dev = torch.device("cuda", 0)
    # two rotating sets, two steps: the second step reuses the workspace the
    # first one filled, on the other image/output set
    wl = bench.DeviceWorkload(ic, cfg, dev, nsets=2)
    for y in wl.y_dev:
        y.fill_(0x5A5A5A5A)
    sh = torch.cuda.current_stream(dev).cuda_stream
    wl.step(0, sh)
    wl.step(1, sh)
    torch.cuda.synchronize(dev)
    assert ic.device_status(sh) == 0
    ref = oracle.conv_fprop(wl.xf, cfg.x_dims, wl.xs, wl.wf, cfg.w_dims, wl.ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode, wl.b, cfg.relu)
    def check(s, what):
        got = wl.output(s)
        if not np.array_equal(got, ref):
            idx = np.argwhere(got != ref)
            first = tuple(idx[0])
            raise AssertionError(f"{name} {what} set {s}: {len(idx)} of {ref.size} outputs differ; first at "
                                 f"{first}: got {got[first]} expected {ref[first]}")

    for s in (0, 1):
        check(s, "conv_fprop")
    # the two halves the convolution-only timing calls
    wl.y_dev[0].fill_(0x5A5A5A5A)
    wl.pack(sh)
    wl.conv(0, sh)
    torch.cuda.synchronize(dev)
    assert ic.device_status(sh) == 0
    check(0, "pack_filter + prepacked")
