"""Seeded synthetic inputs and workload shapes.

This module feeds the same inputs to both sides of every parity check: the
tests and ``bench.py`` call it, and hand its arrays to the oracle and (as
device buffers) to the library.  Neither the library nor its binding imports
it.  It holds no convolution arithmetic: it only draws integers and describes
shapes and memory layouts.

Random numbers come from splitmix64 (Steele, Lea and Flood, "Fast Splittable
Pseudorandom Number Generators", OOPSLA 2014), used as a counter-based
generator: element ``i`` of stream ``key`` is ``mix(key * K0 + (i + 1) * GAMMA)``
with the published splitmix64 finaliser as ``mix``.  Values are produced in the
tensor's *logical* index order (N,C,H,W for images, K,C,R,S for filters) and
only then placed into memory, so one logical tensor is bit-identical in every
layout.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
K0 = np.uint64(0xD1B54A32D192ED03)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

TAG_X, TAG_W, TAG_BIAS, TAG_EXTREME, TAG_EXTREME_SIDE = 1, 2, 3, 4, 5


def splitmix64(key: int, count: int) -> np.ndarray:
    """``count`` outputs of the splitmix64 stream ``key`` (uint64 array)."""
    with np.errstate(over="ignore"):
        i = np.arange(1, count + 1, dtype=np.uint64)
        z = np.uint64(key & 0xFFFFFFFFFFFFFFFF) * K0 + i * GAMMA
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, tag: int) -> int:
    return ((seed & 0xFFFFFFFFFFFF) << 8) | tag


def int8_uniform(seed: int, tag: int, shape: Sequence[int]) -> np.ndarray:
    """int8 uniform on [-128, 127], both ends included: the top byte of each draw."""
    n = int(np.prod(shape))
    z = splitmix64(stream_key(seed, tag), n)
    return (z >> np.uint64(56)).astype(np.uint8).view(np.int8).reshape(shape)


def int8_with_extremes(seed: int, tag: int, shape: Sequence[int], frac: float = 0.1) -> np.ndarray:
    """Uniform int8, then each element independently becomes -128 or 127
    (half each) with probability ``frac``."""
    base = int8_uniform(seed, tag, shape)
    n = base.size
    sel = splitmix64(stream_key(seed, (TAG_EXTREME << 4) | tag), n) >> np.uint64(32)
    side = splitmix64(stream_key(seed, (TAG_EXTREME_SIDE << 4) | tag), n) & np.uint64(1)
    thresh = np.uint64(int(round(frac * 2 ** 32)))
    ext = np.where(side == 0, np.int8(-128), np.int8(127)).astype(np.int8)
    out = np.where((sel < thresh).reshape(shape), ext.reshape(shape), base)
    return out.astype(np.int8)


def int32_uniform(seed: int, tag: int, count: int, lo: int, hi: int) -> np.ndarray:
    """int32 uniform on [lo, hi] (both included) by reduction modulo the span."""
    span = np.uint64(hi - lo + 1)
    z = splitmix64(stream_key(seed, tag), count)
    return ((z % span).astype(np.int64) + lo).astype(np.int32)


# --------------------------------------------------------------------------
# Layouts: logical dims are always [N,C,H,W] (image, output) or [K,C,R,S]
# (filter).  A layout names the memory order from outermost to innermost.
# --------------------------------------------------------------------------
LAYOUT_ORDERS = {
    "NCHW": (0, 1, 2, 3),
    "NHWC": (0, 2, 3, 1),
    "KCRS": (0, 1, 2, 3),
    "KRSC": (0, 2, 3, 1),
}


def packed_strides(dims: Sequence[int], layout: str) -> Tuple[int, ...]:
    """Element strides of a packed tensor with logical ``dims`` in ``layout``."""
    order = LAYOUT_ORDERS[layout]
    strides = [0] * 4
    acc = 1
    for d in reversed(order):
        strides[d] = acc
        acc *= int(dims[d])
    return tuple(strides)


def place(logical: np.ndarray, layout: str, pad_elems: int = 0) -> Tuple[np.ndarray, Tuple[int, ...]]:
    """Lay a logical 4-D array out in ``layout``.

    Returns (flat buffer, element strides).  ``pad_elems`` > 0 appends that many
    unused elements to the innermost run of every row, giving a non-packed but
    legal stride set (used by layout-independence checks).
    """
    order = LAYOUT_ORDERS[layout]
    phys = np.ascontiguousarray(np.transpose(logical, order))
    if pad_elems:
        padded = np.zeros(phys.shape[:-1] + (phys.shape[-1] + pad_elems,), dtype=phys.dtype)
        padded[..., : phys.shape[-1]] = phys
        phys = padded
    pstrides = [0] * 4
    acc = 1
    for i in reversed(range(4)):
        pstrides[i] = acc
        acc *= phys.shape[i]
    strides = [0] * 4
    for i, d in enumerate(order):
        strides[d] = pstrides[i]
    return phys.reshape(-1), tuple(strides)


def gather_logical(flat: np.ndarray, dims: Sequence[int], strides: Sequence[int]) -> np.ndarray:
    """Read a logical 4-D array back out of a flat buffer with given strides."""
    return np.lib.stride_tricks.as_strided(
        flat, shape=tuple(int(d) for d in dims),
        strides=tuple(int(s) * flat.itemsize for s in strides)).copy()


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ConvConfig:
    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    stride: Tuple[int, int] = (1, 1)
    dilation: Tuple[int, int] = (1, 1)
    pre: Tuple[int, int] = (0, 0)
    post: Tuple[int, int] = (0, 0)
    mode: int = 0  # 0 cross-correlation, 1 convolution
    x_layout: str = "NHWC"
    w_layout: str = "KRSC"
    y_layout: str = "NHWC"
    bias: bool = False
    relu: bool = False
    extremes: float = 0.0
    seed: int = 0xC0FFEE

    @property
    def P(self) -> int:
        return (self.H + self.pre[0] + self.post[0] - self.dilation[0] * (self.R - 1) - 1) // self.stride[0] + 1

    @property
    def Q(self) -> int:
        return (self.W + self.pre[1] + self.post[1] - self.dilation[1] * (self.S - 1) - 1) // self.stride[1] + 1

    @property
    def ops(self) -> int:
        """2*N*K*P*Q*C*R*S, padded taps included."""
        return 2 * self.N * self.K * self.P * self.Q * self.C * self.R * self.S

    @property
    def x_dims(self):
        return (self.N, self.C, self.H, self.W)

    @property
    def w_dims(self):
        return (self.K, self.C, self.R, self.S)

    @property
    def y_dims(self):
        return (self.N, self.K, self.P, self.Q)

    def algorithmic_bytes(self) -> int:
        """X + W + Y (+ bias), each touched once."""
        b = self.N * self.C * self.H * self.W + self.K * self.C * self.R * self.S
        b += 4 * self.N * self.K * self.P * self.Q
        if self.bias:
            b += 4 * self.K
        return b


def make_inputs(cfg: ConvConfig, seed: Optional[int] = None):
    """Logical int8 image [N,C,H,W], int8 filter [K,C,R,S], int32 bias [K] or None."""
    s = cfg.seed if seed is None else seed
    if cfg.extremes > 0:
        x = int8_with_extremes(s, TAG_X, cfg.x_dims, cfg.extremes)
        w = int8_with_extremes(s, TAG_W, cfg.w_dims, cfg.extremes)
    else:
        x = int8_uniform(s, TAG_X, cfg.x_dims)
        w = int8_uniform(s, TAG_W, cfg.w_dims)
    b = int32_uniform(s, TAG_BIAS, cfg.K, -(1 << 20), 1 << 20) if cfg.bias else None
    return x, w, b


# The five workloads of the specification, plus the 1x3x32x32 / 64x3x3x3
# correctness shape of "Building a From-Scratch INT8 Strided Convolution
# Kernel" (section "Correctness Testing").  Seeds are 0xC0FFEE + index.
CONFIGS = {
    "c1_tiny_nchw": ConvConfig("c1_tiny_nchw", 1, 1, 5, 5, 1, 3, 3,
                               x_layout="NCHW", w_layout="KCRS", y_layout="NCHW",
                               seed=0xC0FFEE + 0),
    "c2_s2_nhwc": ConvConfig("c2_s2_nhwc", 8, 64, 56, 56, 64, 3, 3, stride=(2, 2),
                             pre=(1, 1), post=(1, 1), seed=0xC0FFEE + 1),
    "c3_3x3_large": ConvConfig("c3_3x3_large", 32, 256, 56, 56, 256, 3, 3,
                               pre=(1, 1), post=(1, 1), seed=0xC0FFEE + 2),
    "c4_1x1_bias_relu": ConvConfig("c4_1x1_bias_relu", 64, 512, 28, 28, 128, 1, 1,
                                   bias=True, relu=True, seed=0xC0FFEE + 3),
    "c5_7x1_dilated_conv": ConvConfig("c5_7x1_dilated_conv", 16, 128, 112, 96, 192, 7, 1,
                                      stride=(2, 1), dilation=(2, 1), pre=(6, 0), post=(5, 0),
                                      mode=1, x_layout="NCHW", w_layout="KCRS",
                                      y_layout="NCHW", extremes=0.1, seed=0xC0FFEE + 4),
    "p4_shape": ConvConfig("p4_shape", 1, 3, 32, 32, 64, 3, 3, x_layout="NCHW",
                           w_layout="KCRS", y_layout="NCHW", seed=0xC0FFEE + 5),
}
