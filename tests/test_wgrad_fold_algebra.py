"""The folded weight gradient's index algebra, checked on the CPU against the
oracle's weight gradient.

With a batch of N <= 32 the library folds T = min(64 // N, Q, 8) columns of
dY into the channels: channel t*N + n of folded tap (p, q2) is
dY[n, k, p, T*q2 + t] (zero from column Q on), and a copy X'' of the image
holds, at column u, channel t*N + n = X[n, c, h, u - pre_w + t*stride_w]
(zero outside X).  The forward convolution of X'' by the folded dY, without
padding along W, with the tap q2 at dilation T*stride_w, the output column s
at stride dilation_w, and along H the forward's stride and dilation
exchanged, must give every dW element.  Here both operands are built with
numpy from those definitions and the folded sum is taken directly; the
oracle's seven-loop weight gradient is the reference (tolerance 0).  The GPU
path is checked against the oracle separately (tests/test_gpu_grad.py)."""
import numpy as np
import pytest

import oracle
import synth


def _folded_dw(x, dy, R, S, pre, stride, dil):
    N, C, H, W = x.shape
    _, K, P, Q = dy.shape
    T = min(64 // N, Q, 8)
    assert T >= 2
    Q2 = -(-Q // T)
    U = T * stride[1] * (Q2 - 1) + dil[1] * (S - 1) + 1
    ch = T * N
    # X''[c, h, u, t*N + n]
    x2 = np.zeros((C, H, U, ch), dtype=np.int64)
    for t in range(T):
        for u in range(U):
            w = u - pre[1] + t * stride[1]
            if 0 <= w < W:
                x2[:, :, u, t * N:(t + 1) * N] = x[:, :, :, w].transpose(1, 2, 0)
    # folded dY[k, p, q2, t*N + n]
    d2 = np.zeros((K, P, Q2, ch), dtype=np.int64)
    for t in range(T):
        for q2 in range(Q2):
            q = T * q2 + t
            if q < Q:
                d2[:, :, q2, t * N:(t + 1) * N] = dy[:, :, :, q].transpose(1, 2, 0)
    dw = np.zeros((K, C, R, S), dtype=np.int64)
    for r in range(R):
        for s in range(S):
            for p in range(P):
                h = dil[0] * r + stride[0] * p - pre[0]
                if not 0 <= h < H:
                    continue
                for q2 in range(Q2):
                    u = dil[1] * s + T * stride[1] * q2
                    dw[:, :, r, s] += d2[:, p, q2, :] @ x2[:, h, u, :].T
    return dw


CASES = [
    # N, C, H, W, K, R, S, pre, post, stride, dil, mode
    (2, 5, 9, 11, 4, 3, 3, (1, 1), (1, 1), (1, 1), (1, 1), 0),
    (8, 3, 12, 13, 5, 3, 3, (1, 1), (1, 0), (2, 2), (1, 1), 0),
    (32, 4, 8, 10, 3, 3, 2, (1, 0), (1, 1), (1, 1), (1, 1), 1),
    (5, 2, 10, 17, 3, 2, 3, (0, 2), (1, 1), (1, 3), (2, 2), 0),
    (3, 3, 9, 20, 2, 3, 3, (2, 3), (0, 1), (2, 1), (1, 3), 1),
    (20, 2, 7, 9, 2, 1, 1, (0, 0), (0, 0), (1, 1), (1, 1), 0),
    # strided along W with several folded columns (Q2 > 1)
    (16, 2, 6, 30, 3, 3, 3, (1, 1), (1, 1), (2, 2), (1, 1), 0),
    (8, 2, 7, 40, 2, 2, 3, (0, 2), (0, 1), (1, 3), (1, 2), 1),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n{}_c{}_{}x{}_s{}{}_d{}{}_m{}".format(
    c[0], c[1], c[2], c[3], *c[9], *c[10], c[11]))
def test_folded_weight_gradient_equals_oracle(case):
    N, C, H, W, K, R, S, pre, post, stride, dil, mode = case
    x = synth.int8_uniform(500 + N, 1, (N, C, H, W))
    yd = oracle.out_dims(x.shape, (K, C, R, S), pre, post, stride, dil)
    dy = synth.int8_uniform(500 + N, 3, yd)
    xf, xs = synth.place(x, "NCHW")
    dyf, dys = synth.place(dy, "NCHW")
    ref = oracle.conv_wgrad(xf, x.shape, xs, dyf, dy.shape, dys, (K, C, R, S), pre, post, stride, dil, mode)
    got = _folded_dw(x.astype(np.int64), dy.astype(np.int64), R, S, pre, stride, dil)
    if mode == 1:  # CONVOLUTION stores tap (r, s) at (R-1-r, S-1-s)
        got = got[:, :, ::-1, ::-1]
    assert np.array_equal(got, ref)
