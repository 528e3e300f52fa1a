/*
 * conv_oracle.c -- plain CPU oracle for INT8 2-D convolution forward
 * propagation with integer accumulation.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the tests, the package smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header or table with the
 * CUDA library.
 *
 * What it computes (cuDNN documentation, "Convolutions", section
 * "Convolution Fprop": response = image * filter, with the argument list of its
 * "Python API" subsection: pre_padding, post_padding, stride, dilation,
 * convolution_mode, compute_data_type), written out as the definition:
 *
 *   for n < N, k < K, p < P, q < Q:
 *     acc = sum over c < C, r < R, s < S of X[n,c,h,w] * W[k,c,r',s']
 *       h = p*stride_h - pre_h + r*dil_h,  w = q*stride_w - pre_w + s*dil_w
 *       terms whose (h, w) lies outside [0,H) x [0,W) are zero (zero padding)
 *       (r', s') = (r, s) in CROSS_CORRELATION, (R-1-r, S-1-s) in CONVOLUTION
 *     Y[n,k,p,q] = acc, then + bias[k] (two's-complement int32 wrap-around),
 *                  then max(0, .) if ReLU is requested.
 *
 *   P = floor((H + pre_h + post_h - dil_h*(R-1) - 1) / stride_h) + 1, and Q
 *   likewise.  This size rule is not printed on the pages; it is the reading
 *   that reproduces both worked shapes they give (5x5 image, 3x3 filter ->
 *   3x3 output in the forum thread "INT8 convolution using cuDNN Python
 *   Frontend"; 32x32 -> 30x30 in "Building a From-Scratch INT8 Strided
 *   Convolution Kernel", section "Correctness Testing").
 *
 * The accumulator is int64 and the loop order is n, k, p, q, c, r, s: the
 * seven-loop shape of the naive loop in "Building a From-Scratch INT8 Strided
 * Convolution Kernel", section "Step 2: Implement the Naive Strided Loop",
 * without that listing's slips (it indexes the filter's output channel with
 * the channel stride, has no padding or dilation, and clamps to int8).  Every
 * element address is sum(index_i * stride_i) over the tensor's own strides,
 * so every layout goes through the same code.
 *
 * An accumulator outside int32 is reported (return value 2) instead of being
 * wrapped: the int32 output type of the compute_data_type=INT32 reading
 * cannot hold it.
 *
 * int8 output (oracle_conv_fprop_i8): the int32 value above (after bias and
 * ReLU) is requantised by an optional rounding arithmetic right shift,
 *   v' = floor((v + 2^(shift-1)) / 2^shift)   for shift > 0,  v' = v for 0,
 * then saturated to [-128, 127].  The saturation is the clamp of the naive
 * loop in "Building a From-Scratch INT8 Strided Convolution Kernel" (section
 * "Step 2") and what the forum thread's int8-typed output holds (its printed
 * words are the int32 truth clamped to int8); the shift is the plainest
 * integer reading of that post's "ReLU and quantization step" roadmap item.
 *
 * Gradients (oracle_conv_dgrad, oracle_conv_wgrad): the same page's sections
 * "Convolution Dgrad" and "Convolution Wgrad" name the operations (data and
 * weight gradient during backpropagation) and their arguments but print no
 * formula; the reading taken is the plain one, the transpose of the forward
 * sum with respect to the image and to the filter, written out below.
 */
#include <stdint.h>
#include <stddef.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_ACC_OUT_OF_INT32 2

typedef struct {
    int64_t pre[2], post[2], stride[2], dil[2];
    int32_t mode;   /* 0 cross-correlation, 1 convolution */
    int32_t relu;   /* 1: max(0, .) after the bias */
} oracle_params;

int64_t oracle_out_extent(int64_t in, int64_t pre, int64_t post, int64_t taps,
                          int64_t dil, int64_t stride) {
    int64_t span = in + pre + post - dil * (taps - 1) - 1;
    if (stride < 1 || span < 0) return 0;
    return span / stride + 1;
}

/* One output element, straight from the definition above. */
static int one_output(const int8_t *x, const int64_t *xd, const int64_t *xs,
                      const int8_t *w, const int64_t *wd, const int64_t *ws,
                      const int32_t *bias, const oracle_params *pp,
                      int64_t n, int64_t k, int64_t p, int64_t q, int32_t *out) {
    const int64_t C = xd[1], H = xd[2], W = xd[3];
    const int64_t R = wd[2], S = wd[3];
    int64_t acc = 0;
    for (int64_t c = 0; c < C; ++c) {
        for (int64_t r = 0; r < R; ++r) {
            for (int64_t s = 0; s < S; ++s) {
                int64_t h = p * pp->stride[0] - pp->pre[0] + r * pp->dil[0];
                int64_t ww = q * pp->stride[1] - pp->pre[1] + s * pp->dil[1];
                if (h < 0 || h >= H || ww < 0 || ww >= W) continue; /* zero padding */
                int64_t rf = pp->mode ? (R - 1 - r) : r;
                int64_t sf = pp->mode ? (S - 1 - s) : s;
                int64_t xv = x[n * xs[0] + c * xs[1] + h * xs[2] + ww * xs[3]];
                int64_t wv = w[k * ws[0] + c * ws[1] + rf * ws[2] + sf * ws[3]];
                acc += xv * wv;
            }
        }
    }
    if (acc > INT32_MAX || acc < INT32_MIN) return ORACLE_ACC_OUT_OF_INT32;
    int32_t v = (int32_t)acc;
    if (bias) v = (int32_t)((uint32_t)v + (uint32_t)bias[k]);
    if (pp->relu && v < 0) v = 0;
    *out = v;
    return ORACLE_OK;
}

static int check_args(const int64_t *xd, const int64_t *wd, const int64_t *yd,
                      const oracle_params *pp) {
    if (xd[1] != wd[1]) return ORACLE_BAD_ARGS;
    if (yd[0] != xd[0] || yd[1] != wd[0]) return ORACLE_BAD_ARGS;
    for (int i = 0; i < 2; ++i)
        if (pp->stride[i] < 1 || pp->dil[i] < 1 || pp->pre[i] < 0 || pp->post[i] < 0)
            return ORACLE_BAD_ARGS;
    if (yd[2] != oracle_out_extent(xd[2], pp->pre[0], pp->post[0], wd[2], pp->dil[0], pp->stride[0]))
        return ORACLE_BAD_ARGS;
    if (yd[3] != oracle_out_extent(xd[3], pp->pre[1], pp->post[1], wd[3], pp->dil[1], pp->stride[1]))
        return ORACLE_BAD_ARGS;
    return ORACLE_OK;
}

/* Full output.  x: logical [N,C,H,W]; w: [K,C,R,S]; y: [N,K,P,Q]; strides in
 * elements.  bias may be NULL.  The (n, k) pairs are independent, so they are
 * shared out over OpenMP threads when the build enables it. */
int oracle_conv_fprop(const int8_t *x, const int64_t *xd, const int64_t *xs,
                      const int8_t *w, const int64_t *wd, const int64_t *ws,
                      int32_t *y, const int64_t *yd, const int64_t *ys,
                      const int32_t *bias, const oracle_params *pp) {
    int rc = check_args(xd, wd, yd, pp);
    if (rc) return rc;
    const int64_t N = yd[0], K = yd[1], P = yd[2], Q = yd[3];
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            for (int64_t p = 0; p < P; ++p) {
                for (int64_t q = 0; q < Q; ++q) {
                    int32_t v = 0;
                    if (one_output(x, xd, xs, w, wd, ws, bias, pp, n, k, p, q, &v)) bad = 1;
                    y[n * ys[0] + k * ys[1] + p * ys[2] + q * ys[3]] = v;
                }
            }
        }
    }
    return bad ? ORACLE_ACC_OUT_OF_INT32 : ORACLE_OK;
}

/* int8 output: v (int32, after bias and ReLU) -> rounding shift -> clamp. */
static int8_t requant_i8(int32_t v, int32_t shift) {
    int64_t t = v;
    if (shift > 0) {
        t += (int64_t)1 << (shift - 1);
        /* floor division by 2^shift, also for negative t */
        t = (t >= 0) ? (t >> shift) : -((-t + ((int64_t)1 << shift) - 1) >> shift);
    }
    if (t > 127) t = 127;
    if (t < -128) t = -128;
    return (int8_t)t;
}

int oracle_conv_fprop_i8(const int8_t *x, const int64_t *xd, const int64_t *xs,
                         const int8_t *w, const int64_t *wd, const int64_t *ws,
                         int8_t *y, const int64_t *yd, const int64_t *ys,
                         const int32_t *bias, const oracle_params *pp, int32_t shift) {
    int rc = check_args(xd, wd, yd, pp);
    if (rc) return rc;
    if (shift < 0 || shift > 31) return ORACLE_BAD_ARGS;
    const int64_t N = yd[0], K = yd[1], P = yd[2], Q = yd[3];
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t k = 0; k < K; ++k) {
            for (int64_t p = 0; p < P; ++p) {
                for (int64_t q = 0; q < Q; ++q) {
                    int32_t v = 0;
                    if (one_output(x, xd, xs, w, wd, ws, bias, pp, n, k, p, q, &v)) bad = 1;
                    y[n * ys[0] + k * ys[1] + p * ys[2] + q * ys[3]] = requant_i8(v, shift);
                }
            }
        }
    }
    return bad ? ORACLE_ACC_OUT_OF_INT32 : ORACLE_OK;
}

/* Selected outputs only: idx holds count rows of (n, k, p, q); out[i] gets
 * Y at row i.  Used at sizes where the full output is too slow on the CPU. */
int oracle_conv_fprop_points(const int8_t *x, const int64_t *xd, const int64_t *xs,
                             const int8_t *w, const int64_t *wd, const int64_t *ws,
                             const int64_t *yd, const int32_t *bias,
                             const oracle_params *pp, const int64_t *idx,
                             int64_t count, int32_t *out) {
    int rc = check_args(xd, wd, yd, pp);
    if (rc) return rc;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t i = 0; i < count; ++i) {
        const int64_t *t = idx + 4 * i;
        if (t[0] < 0 || t[0] >= yd[0] || t[1] < 0 || t[1] >= yd[1] ||
            t[2] < 0 || t[2] >= yd[2] || t[3] < 0 || t[3] >= yd[3]) {
            bad |= 1;
            continue;
        }
        if (one_output(x, xd, xs, w, wd, ws, bias, pp, t[0], t[1], t[2], t[3], out + i)) bad |= 2;
    }
    if (bad & 1) return ORACLE_BAD_ARGS;
    return bad ? ORACLE_ACC_OUT_OF_INT32 : ORACLE_OK;
}

/*
 * Data gradient (cuDNN "Convolutions", section "Convolution Dgrad": the
 * gradient with respect to the image during backpropagation, from the loss
 * gradient dY -- the "loss" argument, logical [N,K,P,Q] -- and the filter).
 * The fprop above is linear in X, so the data gradient is its transpose
 * applied to dY: every fprop term X[n,c,h,w] * W[k,c,r',s'] that fed
 * Y[n,k,p,q] sends dY[n,k,p,q] * W[k,c,r',s'] back to position (h, w):
 *
 *   dX[n,c,h,w] = sum over k < K, r < R, s < S of dY[n,k,p,q] * W[k,c,r',s']
 *     where p = (h + pre_h - r*dil_h) / stride_h and q likewise, counted only
 *     when the division is exact and 0 <= p < P, 0 <= q < Q;
 *     (r', s') as in fprop (flipped in CONVOLUTION mode).
 *
 * The image size H x W is that of dX's descriptor (with a stride above 1
 * several H give the same P); dY's P, Q must be the fprop output size of it.
 * No bias, ReLU or int8 output: the result is the int32 gradient.  The
 * accumulator is int64 and one outside int32 is reported, as in fprop.
 */
static int check_grad_args(const int64_t *xd, const int64_t *wd, const int64_t *yd,
                           const oracle_params *pp) {
    if (pp->relu) return ORACLE_BAD_ARGS;
    return check_args(xd, wd, yd, pp);
}

int oracle_conv_dgrad(const int8_t *dy, const int64_t *yd, const int64_t *ys,
                      const int8_t *w, const int64_t *wd, const int64_t *ws,
                      int32_t *dx, const int64_t *xd, const int64_t *xs,
                      const oracle_params *pp) {
    int rc = check_grad_args(xd, wd, yd, pp);
    if (rc) return rc;
    const int64_t N = xd[0], C = xd[1], H = xd[2], W = xd[3];
    const int64_t K = wd[0], R = wd[2], S = wd[3], P = yd[2], Q = yd[3];
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t c = 0; c < C; ++c) {
            for (int64_t h = 0; h < H; ++h) {
                for (int64_t ww = 0; ww < W; ++ww) {
                    int64_t acc = 0;
                    for (int64_t k = 0; k < K; ++k) {
                        for (int64_t r = 0; r < R; ++r) {
                            int64_t th = h + pp->pre[0] - r * pp->dil[0];
                            if (th < 0 || th % pp->stride[0]) continue;
                            int64_t p = th / pp->stride[0];
                            if (p >= P) continue;
                            for (int64_t s = 0; s < S; ++s) {
                                int64_t tw = ww + pp->pre[1] - s * pp->dil[1];
                                if (tw < 0 || tw % pp->stride[1]) continue;
                                int64_t q = tw / pp->stride[1];
                                if (q >= Q) continue;
                                int64_t rf = pp->mode ? (R - 1 - r) : r;
                                int64_t sf = pp->mode ? (S - 1 - s) : s;
                                int64_t gv = dy[n * ys[0] + k * ys[1] + p * ys[2] + q * ys[3]];
                                int64_t wv = w[k * ws[0] + c * ws[1] + rf * ws[2] + sf * ws[3]];
                                acc += gv * wv;
                            }
                        }
                    }
                    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
                    dx[n * xs[0] + c * xs[1] + h * xs[2] + ww * xs[3]] = (int32_t)acc;
                }
            }
        }
    }
    return bad ? ORACLE_ACC_OUT_OF_INT32 : ORACLE_OK;
}

/*
 * Weight gradient (cuDNN "Convolutions", section "Convolution Wgrad": the
 * gradient with respect to the filter, from the image and the loss gradient
 * dY).  fprop is linear in W, and W[k,c,r',s'] multiplies X[n,c,h,w] in the
 * term feeding Y[n,k,p,q], so:
 *
 *   dW[k,c,r',s'] = sum over n < N, p < P, q < Q of dY[n,k,p,q] * X[n,c,h,w]
 *     h = p*stride_h - pre_h + r*dil_h, w = q*stride_w - pre_w + s*dil_w,
 *     zero outside the image; (r', s') = (r, s), or (R-1-r, S-1-s) in
 *     CONVOLUTION mode.
 *
 * R x S is that of dW's descriptor.  int64 accumulator, int32 result.
 */
int oracle_conv_wgrad(const int8_t *x, const int64_t *xd, const int64_t *xs,
                      const int8_t *dy, const int64_t *yd, const int64_t *ys,
                      int32_t *dw, const int64_t *wd, const int64_t *ws,
                      const oracle_params *pp) {
    int rc = check_grad_args(xd, wd, yd, pp);
    if (rc) return rc;
    const int64_t N = xd[0], C = xd[1], H = xd[2], W = xd[3];
    const int64_t K = wd[0], R = wd[2], S = wd[3], P = yd[2], Q = yd[3];
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(| : bad)
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t c = 0; c < C; ++c) {
            for (int64_t r = 0; r < R; ++r) {
                for (int64_t s = 0; s < S; ++s) {
                    int64_t acc = 0;
                    for (int64_t n = 0; n < N; ++n) {
                        for (int64_t p = 0; p < P; ++p) {
                            int64_t h = p * pp->stride[0] - pp->pre[0] + r * pp->dil[0];
                            if (h < 0 || h >= H) continue;
                            for (int64_t q = 0; q < Q; ++q) {
                                int64_t ww = q * pp->stride[1] - pp->pre[1] + s * pp->dil[1];
                                if (ww < 0 || ww >= W) continue;
                                int64_t gv = dy[n * ys[0] + k * ys[1] + p * ys[2] + q * ys[3]];
                                int64_t xv = x[n * xs[0] + c * xs[1] + h * xs[2] + ww * xs[3]];
                                acc += gv * xv;
                            }
                        }
                    }
                    int64_t rf = pp->mode ? (R - 1 - r) : r;
                    int64_t sf = pp->mode ? (S - 1 - s) : s;
                    if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
                    dw[k * ws[0] + c * ws[1] + rf * ws[2] + sf * ws[3]] = (int32_t)acc;
                }
            }
        }
    }
    return bad ? ORACLE_ACC_OUT_OF_INT32 : ORACLE_OK;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP), and a
 * way to change it (used to time the oracle on one core). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
