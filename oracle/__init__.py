"""CPU oracle for INT8 conv2d forward propagation with int32 results, and for
the data and weight gradients of the same convolution.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package; only ``tests/``, the package smoke check
and the CPU-baseline leg of ``bench.py`` do.  It shares no code with the CUDA
path.

Contents
--------
* ``conv_fprop`` / ``conv_fprop_points``: ctypes front ends to the plain C
  seven-loop definition in ``conv_oracle.c`` (int64 accumulation).
* ``conv_fprop_pyint``: the same definition over Python integers, for tiny
  brute-force cases.
* ``out_extent``: the output-size rule.
* ``saturate_int8`` / ``pack_int8_words``: the int8-output reading of the
  forum thread "INT8 convolution using cuDNN Python Frontend" (its printed
  cuDNN words are the int32 truth clamped to int8, four bytes to a word).
* ``conv_fprop(..., out_int8=True, out_shift=s)``: the int8 output (rounding
  right shift, then saturation).
* ``conv_dgrad`` / ``conv_wgrad``: the data and weight gradients ("Convolutions",
  sections "Convolution Dgrad" and "Convolution Wgrad"), written in C as the
  transposes of the forward sum; ``grads_pyint`` derives both over Python
  integers by the chain rule applied term by term to the forward definition.
* ``worst_case_abs``: the accumulator bound |acc| <= C*R*S*2^14.

Parity status: every function here is pinned by tests in
``tests/test_oracle.py`` except that the forum thread's nine truth values
cannot be recomputed (its inputs were drawn unseeded and never printed):
that single example is "parity unpinned" as a convolution, and is used only to
pin ``saturate_int8`` / ``pack_int8_words``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "conv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


class _Params(ctypes.Structure):
    _fields_ = [("pre", ctypes.c_int64 * 2), ("post", ctypes.c_int64 * 2),
                ("stride", ctypes.c_int64 * 2), ("dil", ctypes.c_int64 * 2),
                ("mode", ctypes.c_int32), ("relu", ctypes.c_int32)]


def build(force: bool = False) -> str:
    """Compile conv_oracle.c into liboracle.so (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_conv_fprop.restype = ctypes.c_int
    lib.oracle_conv_fprop.argtypes = [ctypes.c_void_p, i64p, i64p, ctypes.c_void_p, i64p, i64p,
                                      ctypes.c_void_p, i64p, i64p, ctypes.c_void_p,
                                      ctypes.POINTER(_Params)]
    lib.oracle_conv_fprop_points.restype = ctypes.c_int
    lib.oracle_conv_fprop_points.argtypes = [ctypes.c_void_p, i64p, i64p, ctypes.c_void_p, i64p,
                                             i64p, i64p, ctypes.c_void_p,
                                             ctypes.POINTER(_Params), i64p, ctypes.c_int64,
                                             ctypes.c_void_p]
    lib.oracle_conv_fprop_i8.restype = ctypes.c_int
    lib.oracle_conv_fprop_i8.argtypes = [ctypes.c_void_p, i64p, i64p, ctypes.c_void_p, i64p, i64p,
                                         ctypes.c_void_p, i64p, i64p, ctypes.c_void_p,
                                         ctypes.POINTER(_Params), ctypes.c_int32]
    for name in ("oracle_conv_dgrad", "oracle_conv_wgrad"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, i64p, i64p, ctypes.c_void_p, i64p, i64p, ctypes.c_void_p, i64p, i64p,
                      ctypes.POINTER(_Params)]
    lib.oracle_out_extent.restype = ctypes.c_int64
    lib.oracle_out_extent.argtypes = [ctypes.c_int64] * 6
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(build())
    return _lib


def use_library(path: Optional[str]) -> None:
    """Point this module at another build of the oracle (``None``: the default
    build).  Used only by the test that plants mistakes in a copy of the C
    source to show that the pins catch them."""
    global _lib
    _lib = None if path is None else _bind(path)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the OpenMP loops use from now on (timing only; results do not
    depend on it)."""
    _load().oracle_set_num_threads(int(n))


def _i64(vals: Sequence[int]):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def _params(pre, post, stride, dilation, mode, relu) -> _Params:
    p = _Params()
    for i in range(2):
        p.pre[i], p.post[i] = int(pre[i]), int(post[i])
        p.stride[i], p.dil[i] = int(stride[i]), int(dilation[i])
    p.mode, p.relu = int(mode), int(bool(relu))
    return p


def out_extent(size: int, pre: int, post: int, taps: int, dil: int, stride: int) -> int:
    """floor((size + pre + post - dil*(taps-1) - 1) / stride) + 1, or 0 if empty."""
    return int(_load().oracle_out_extent(size, pre, post, taps, dil, stride))


def out_dims(x_dims, w_dims, pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1)):
    N, C, H, W = x_dims
    K, _, R, S = w_dims
    return (N, K, out_extent(H, pre[0], post[0], R, dilation[0], stride[0]),
            out_extent(W, pre[1], post[1], S, dilation[1], stride[1]))


def conv_fprop(x_flat: np.ndarray, x_dims, x_strides, w_flat: np.ndarray, w_dims, w_strides,
               pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode: int = 0,
               bias: Optional[np.ndarray] = None, relu: bool = False,
               y_strides=None, out_int8: bool = False, out_shift: int = 0) -> np.ndarray:
    """Full convolution.  Inputs are flat buffers plus logical dims and element
    strides.  Returns the logical output [N,K,P,Q] (packed NCHW) unless
    ``y_strides`` is given, in which case the flat buffer in that layout is
    returned.  The output is int32, or with ``out_int8`` int8 after the
    rounding right shift by ``out_shift`` and saturation."""
    lib = _load()
    x_flat = np.ascontiguousarray(x_flat, dtype=np.int8)
    w_flat = np.ascontiguousarray(w_flat, dtype=np.int8)
    yd = out_dims(x_dims, w_dims, pre, post, stride, dilation)
    if y_strides is None:
        y_strides = (yd[1] * yd[2] * yd[3], yd[2] * yd[3], yd[3], 1)
    ysize = 1 + sum((d - 1) * s for d, s in zip(yd, y_strides)) if min(yd) > 0 else 0
    y = np.zeros(max(ysize, 1), dtype=np.int8 if out_int8 else np.int32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.int32)
    p = _params(pre, post, stride, dilation, mode, relu)
    if out_int8:
        rc = lib.oracle_conv_fprop_i8(x_flat.ctypes.data, _i64(x_dims), _i64(x_strides),
                                      w_flat.ctypes.data, _i64(w_dims), _i64(w_strides),
                                      y.ctypes.data, _i64(yd), _i64(y_strides),
                                      None if b is None else b.ctypes.data, ctypes.byref(p), int(out_shift))
    else:
        rc = lib.oracle_conv_fprop(x_flat.ctypes.data, _i64(x_dims), _i64(x_strides),
                                   w_flat.ctypes.data, _i64(w_dims), _i64(w_strides),
                                   y.ctypes.data, _i64(yd), _i64(y_strides),
                                   None if b is None else b.ctypes.data, ctypes.byref(p))
    if rc == 2:
        raise OverflowError("accumulator outside int32")
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    if tuple(y_strides) == (yd[1] * yd[2] * yd[3], yd[2] * yd[3], yd[3], 1):
        return y[: int(np.prod(yd))].reshape(yd)
    return y


def conv_fprop_points(x_flat, x_dims, x_strides, w_flat, w_dims, w_strides, points: np.ndarray,
                      pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode: int = 0,
                      bias: Optional[np.ndarray] = None, relu: bool = False) -> np.ndarray:
    """Y at the given (n, k, p, q) rows of ``points`` (int64 array [count, 4])."""
    lib = _load()
    x_flat = np.ascontiguousarray(x_flat, dtype=np.int8)
    w_flat = np.ascontiguousarray(w_flat, dtype=np.int8)
    pts = np.ascontiguousarray(points, dtype=np.int64).reshape(-1, 4)
    yd = out_dims(x_dims, w_dims, pre, post, stride, dilation)
    out = np.zeros(len(pts), dtype=np.int32)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.int32)
    p = _params(pre, post, stride, dilation, mode, relu)
    rc = lib.oracle_conv_fprop_points(
        x_flat.ctypes.data, _i64(x_dims), _i64(x_strides), w_flat.ctypes.data, _i64(w_dims),
        _i64(w_strides), _i64(yd), None if b is None else b.ctypes.data, ctypes.byref(p),
        pts.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(pts), out.ctypes.data)
    if rc == 2:
        raise OverflowError("accumulator outside int32")
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return out


def conv_fprop_pyint(x, w, pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode=0,
                     bias=None, relu=False):
    """The definition over Python integers on logical nested arrays (tiny cases only)."""
    N, C, H, W = x.shape
    K, _, R, S = w.shape
    _, _, P, Q = out_dims(x.shape, w.shape, pre, post, stride, dilation)
    y = [[[[0] * Q for _ in range(P)] for _ in range(K)] for _ in range(N)]
    for n in range(N):
        for k in range(K):
            for p in range(P):
                for q in range(Q):
                    acc = 0
                    for c in range(C):
                        for r in range(R):
                            for s in range(S):
                                h = p * stride[0] - pre[0] + r * dilation[0]
                                ww = q * stride[1] - pre[1] + s * dilation[1]
                                if 0 <= h < H and 0 <= ww < W:
                                    rf, sf = (R - 1 - r, S - 1 - s) if mode else (r, s)
                                    acc += int(x[n, c, h, ww]) * int(w[k, c, rf, sf])
                    if bias is not None:
                        acc = (acc + int(bias[k]) + 2 ** 31) % 2 ** 32 - 2 ** 31
                    if relu:
                        acc = max(acc, 0)
                    y[n][k][p][q] = acc
    return np.array(y, dtype=np.int64).reshape(N, K, P, Q)


def _packed(dims):
    return (dims[1] * dims[2] * dims[3], dims[2] * dims[3], dims[3], 1)


def conv_dgrad(dy_flat, dy_dims, dy_strides, w_flat, w_dims, w_strides, x_dims,
               pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode: int = 0) -> np.ndarray:
    """Data gradient dX (logical [N,C,H,W] int32, packed NCHW) of the image of
    size ``x_dims`` from the loss gradient dY [N,K,P,Q] and the filter."""
    lib = _load()
    dy_flat = np.ascontiguousarray(dy_flat, dtype=np.int8)
    w_flat = np.ascontiguousarray(w_flat, dtype=np.int8)
    xs = _packed(x_dims)
    dx = np.zeros(max(int(np.prod(x_dims)), 1), dtype=np.int32)
    p = _params(pre, post, stride, dilation, mode, False)
    rc = lib.oracle_conv_dgrad(dy_flat.ctypes.data, _i64(dy_dims), _i64(dy_strides), w_flat.ctypes.data,
                               _i64(w_dims), _i64(w_strides), dx.ctypes.data, _i64(x_dims), _i64(xs),
                               ctypes.byref(p))
    if rc == 2:
        raise OverflowError("accumulator outside int32")
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return dx[: int(np.prod(x_dims))].reshape(x_dims)


def conv_wgrad(x_flat, x_dims, x_strides, dy_flat, dy_dims, dy_strides, w_dims,
               pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode: int = 0) -> np.ndarray:
    """Weight gradient dW (logical [K,C,R,S] int32, packed KCRS) of a filter of
    size ``w_dims`` from the image and the loss gradient dY [N,K,P,Q]."""
    lib = _load()
    x_flat = np.ascontiguousarray(x_flat, dtype=np.int8)
    dy_flat = np.ascontiguousarray(dy_flat, dtype=np.int8)
    ws = _packed(w_dims)
    dw = np.zeros(max(int(np.prod(w_dims)), 1), dtype=np.int32)
    p = _params(pre, post, stride, dilation, mode, False)
    rc = lib.oracle_conv_wgrad(x_flat.ctypes.data, _i64(x_dims), _i64(x_strides), dy_flat.ctypes.data,
                               _i64(dy_dims), _i64(dy_strides), dw.ctypes.data, _i64(w_dims), _i64(ws),
                               ctypes.byref(p))
    if rc == 2:
        raise OverflowError("accumulator outside int32")
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return dw[: int(np.prod(w_dims))].reshape(w_dims)


def grads_pyint(x, w, dy, pre=(0, 0), post=(0, 0), stride=(1, 1), dilation=(1, 1), mode=0):
    """dX and dW over Python integers (tiny cases only), by walking every term
    X[n,c,h,w] * W[k,c,r',s'] of the forward sum and sending dY[n,k,p,q] back
    along it: the chain rule applied to the definition term by term."""
    N, C, H, W = x.shape
    K, _, R, S = w.shape
    _, _, P, Q = out_dims(x.shape, w.shape, pre, post, stride, dilation)
    dx = [[[[0] * W for _ in range(H)] for _ in range(C)] for _ in range(N)]
    dw = [[[[0] * S for _ in range(R)] for _ in range(C)] for _ in range(K)]
    for n in range(N):
        for k in range(K):
            for p in range(P):
                for q in range(Q):
                    g = int(dy[n, k, p, q])
                    for c in range(C):
                        for r in range(R):
                            for s in range(S):
                                h = p * stride[0] - pre[0] + r * dilation[0]
                                ww = q * stride[1] - pre[1] + s * dilation[1]
                                if 0 <= h < H and 0 <= ww < W:
                                    rf, sf = (R - 1 - r, S - 1 - s) if mode else (r, s)
                                    dx[n][c][h][ww] += g * int(w[k, c, rf, sf])
                                    dw[k][c][rf][sf] += g * int(x[n, c, h, ww])
    return np.array(dx, dtype=np.int64), np.array(dw, dtype=np.int64)


def worst_case_abs(C: int, R: int, S: int, bias_abs: int = 0) -> int:
    """Largest |accumulator| any int8 input can produce: C*R*S*(-128)^2 (+|bias|)."""
    return C * R * S * 128 * 128 + bias_abs


def saturate_int8(y: np.ndarray) -> np.ndarray:
    """Clamp int32 results to [-128, 127] (the int8-output reading)."""
    return np.clip(np.asarray(y, dtype=np.int64), -128, 127).astype(np.int8)


def pack_int8_words(b: np.ndarray) -> np.ndarray:
    """Little-endian packing of an int8 sequence into int32 words, zero-filled
    to a multiple of four bytes (how an int8 result lands in an int32 buffer)."""
    raw = np.asarray(b, dtype=np.int8).reshape(-1).view(np.uint8)
    pad = (-len(raw)) % 4
    raw = np.concatenate([raw, np.zeros(pad, dtype=np.uint8)])
    return raw.view("<i4").astype(np.int32)
