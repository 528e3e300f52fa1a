"""Exactness of the tensor-core route where it could fail.

The tensor-core kernel forms int8 products on the f16 MMA path and sums them
in f32 tensor-memory accumulators, in groups of at most 1024 products, which
it then adds in int32.  That is exact only if each f32 sum keeps every bit of
its 24-bit significand while |sum| < 2^24.  Sums whose low bits are zero
(all products multiples of 2^7 or 2^14) cannot show a dropped last bit, and
random signs keep partial sums far below 2^23.  The cases here put ODD
products onto accumulators between 2^23 and 2^24:

* every operand -127: each product is 16129 (odd) and 1024 of them sum to
  16,516,096;
* inside each 16-product slice of the reduction (one K=16 MMA step) fifteen
  products of 2^14 and one of +1 or -1, the odd one at every position of the
  slice in turn, so that the last product of every 1024-product group is one
  of them;
* all -127 with one product per pixel replaced by an odd one of size 127, its
  position running over the whole reduction (first, middle and group end);
* same-sign random operands in [-128, -97] (products 9409..16384 of both
  parities; partial sums climb to ~1.4e7 inside each group).

Each is compared element by element with the CPU oracle (tolerance 0), on
both producers (TMA im2col and global loads), on 128- and 256-column tiles
and on the cut-reduction route (few tiles with long reductions).
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TWO24 = 1 << 24


@pytest.fixture(scope="module")
def ic():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import int8_conv2d_fprop_gb300 as m
    torch.cuda.set_device(0)
    return m


def _run(ic, cfg, x, w, algo):
    xf, xs = synth.place(x, cfg.x_layout)
    wf, ws = synth.place(w, cfg.w_layout)
    xt = torch.as_strided(torch.from_numpy(xf).cuda(), cfg.x_dims, xs)
    wt = torch.as_strided(torch.from_numpy(wf).cuda(), cfg.w_dims, ws)
    y = ic.conv_fprop(xt, wt, pre_padding=cfg.pre, post_padding=cfg.post, stride=cfg.stride,
                      dilation=cfg.dilation, mode=cfg.mode, algo=algo)
    torch.cuda.synchronize()
    assert ic.device_status() == 0
    ref = oracle.conv_fprop(xf, cfg.x_dims, xs, wf, cfg.w_dims, ws, cfg.pre, cfg.post, cfg.stride,
                            cfg.dilation, cfg.mode)
    return y.cpu().numpy(), ref


def _assert_equal(got, ref, what):
    if not np.array_equal(got, ref):
        idx = np.argwhere(got != ref)
        first = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {ref.size} outputs differ; first at {first}: "
                             f"got {got[first]} expected {ref[first]} (diff {int(got[first]) - int(ref[first])})")


ALGOS = [1, 4]  # tensor cores: TMA im2col producer, global-load producer


def _shapes():
    C = synth.ConvConfig
    return [
        # one group of exactly 1024 products per output (16 k-steps of 64 channels)
        C("crs1024_k64", 2, 1024, 9, 9, 64, 1, 1),
        # two groups of 1024, 256-column tiles (K > 128)
        C("crs2048_k200", 1, 2048, 8, 8, 200, 1, 1),
        # 3x3, C=256: interior outputs reduce over 2304 products (three groups
        # of 768), 128-column tiles
        C("crs2304_3x3", 2, 256, 8, 8, 96, 3, 3, pre=(1, 1), post=(1, 1)),
        # few tiles, 64 k-steps: the reduction is cut into runs that different
        # CTAs compute and the reduction kernel adds
        C("cut_runs_crs4096", 1, 4096, 8, 8, 64, 1, 1),
    ]


def _all_m127(cfg):
    return (np.full(cfg.x_dims, -127, dtype=np.int8), np.full(cfg.w_dims, -127, dtype=np.int8))


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("cfg", _shapes(), ids=lambda c: c.name)
def test_all_minus_127(ic, cfg, algo):
    x, w = _all_m127(cfg)
    got, ref = _run(ic, cfg, x, w, algo)
    crs = cfg.C * cfg.R * cfg.S
    assert int(ref.max()) == crs * 16129  # an interior output reduces over every tap
    # the kernel's groups hold 12 or 16 k-steps of 64 channels here: 768 or
    # 1024 products of 16129, i.e. 12.4e6 or 16.5e6, both in [2^23, 2^24)
    assert (TWO24 >> 1) <= 768 * 16129 and 1024 * 16129 < TWO24
    _assert_equal(got, ref, f"all -127 {cfg.name} algo {algo}")


def _slice_pattern(cfg, seed):
    """Fifteen products of 2^14 and one of +-1 in every 16-channel slice of
    the reduction but the first (16 products of 2^14), so that each tap adds
    an odd number of odd terms; the odd product sits at position (slice
    index mod 16)."""
    rng = np.random.default_rng(seed)
    x = np.full(cfg.x_dims, -128, dtype=np.int8)
    w = np.full(cfg.w_dims, -128, dtype=np.int8)
    slices = cfg.C // 16
    for t in range(1, slices):
        c = 16 * t + (t % 16)
        x[:, c] = rng.choice(np.array([-1, 1], dtype=np.int8), size=x[:, c].shape)
        w[:, c] = rng.choice(np.array([-1, 1], dtype=np.int8), size=w[:, c].shape)
    return x, w


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("cfg", _shapes(), ids=lambda c: c.name)
def test_one_odd_product_per_mma_slice(ic, cfg, algo):
    x, w = _slice_pattern(cfg, seed=cfg.C + cfg.K)
    got, ref = _run(ic, cfg, x, w, algo)
    # interior: one slice of 16 * 2^14 and C/16 - 1 slices of 15 * 2^14 +- 1
    # per tap; an odd count of +-1 terms per tap
    slices = cfg.C // 16
    top = cfg.R * cfg.S * (16 * 16384 + (slices - 1) * 15 * 16384)
    assert top - cfg.R * cfg.S * (slices - 1) <= int(ref.max()) <= top + cfg.R * cfg.S * (slices - 1)
    assert np.any(ref % 2 != 0)
    _assert_equal(got, ref, f"slice pattern {cfg.name} algo {algo}")


def _moving_odd_term(cfg, seed):
    """All -127, except that at pixel (n, h, w) channel c = (pixel index * 37)
    mod C is +-1: one product of -+127 per tap whose position runs over the
    whole channel range, group ends included."""
    rng = np.random.default_rng(seed)
    x = np.full(cfg.x_dims, -127, dtype=np.int8)
    w = np.full(cfg.w_dims, -127, dtype=np.int8)
    N, C, H, W = cfg.x_dims
    idx = np.arange(N * H * W)
    ch = (idx * 37) % C
    # force the first, last and group-end channels in
    for i, c in enumerate([0, C - 1, 1023 % C, 1024 % C, 63, 64]):
        if i < len(ch):
            ch[i] = c
    n, hw = np.divmod(idx, H * W)
    h, ww = np.divmod(hw, W)
    x[n, ch, h, ww] = rng.choice(np.array([-1, 1], dtype=np.int8), size=idx.size)
    return x, w


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("cfg", _shapes(), ids=lambda c: c.name)
def test_odd_term_at_every_reduction_position(ic, cfg, algo):
    x, w = _moving_odd_term(cfg, seed=7 + cfg.C)
    got, ref = _run(ic, cfg, x, w, algo)
    _assert_equal(got, ref, f"moving odd term {cfg.name} algo {algo}")


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("cfg", _shapes() + [
    # the 3x3 workload's channel count and padding at two images of 56 x 56
    synth.ConvConfig("c3_shape_n2", 2, 256, 56, 56, 256, 3, 3, pre=(1, 1), post=(1, 1)),
], ids=lambda c: c.name)
def test_same_sign_random_near_two_to_24(ic, cfg, algo):
    rng = np.random.default_rng(cfg.C * 3 + cfg.H)
    x = rng.integers(-128, -96, size=cfg.x_dims, endpoint=False).astype(np.int8)
    w = rng.integers(-128, -96, size=cfg.w_dims, endpoint=False).astype(np.int8)
    got, ref = _run(ic, cfg, x, w, algo)
    crs = cfg.C * cfg.R * cfg.S
    # a full group's partial sum climbs past 2^23: the smallest product is 97^2
    assert min(crs, 1024) * 97 * 97 > (TWO24 >> 1) or crs < 1024
    assert np.any(ref % 2 != 0)
    _assert_equal(got, ref, f"same-sign random {cfg.name} algo {algo}")
