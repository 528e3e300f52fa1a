// desc.cpp -- tensor descriptors, the stride calculator and the validator.
//
// Descriptors follow the forum thread "INT8 convolution using cuDNN Python
// Frontend": logical dims plus one element stride per logical dim.  That
// thread's failure (int32 truth values replaced by int8-saturated bytes packed
// into the int32 buffer) came from an output whose type was left to default to
// the graph's int8 I/O type, next to stride sets that the reply called
// inconsistent.  The validator below therefore requires the output type to be
// given as INT32 and checks every stride set for positivity, non-aliasing and
// fit inside the caller's buffer.
#include <algorithm>
#include <cstring>

#include "internal.h"

namespace i8c {

static bool mul_ok(int64_t a, int64_t b, int64_t *out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / 4 / a) return false;
    *out = a * b;
    return true;
}

int64_t desc_extent_elems(const conv_tensor_desc *d) {
    int64_t hi = 0;
    for (int i = 0; i < 4; ++i) {
        if (d->dims[i] == 0) return 0;
        hi += (d->dims[i] - 1) * d->strides[i];
    }
    return hi + 1;
}

static int64_t elem_size(int32_t dtype) { return dtype == CONV_INT32 ? 4 : 1; }

// Checks one descriptor: rank, type, dims >= min_dim, strides of non-unit
// dims positive, no two index tuples mapping to one element, extent inside
// capacity_bytes, and every offset inside the library's int64 index range.
static conv_status check_desc(const conv_tensor_desc *d, int32_t dtype, const int64_t min_dims[4]) {
    if (!d) return CONV_ERR_NULL_PTR;
    if (d->rank != 4) return CONV_ERR_RANK;
    if (d->dtype != dtype) return CONV_ERR_DTYPE;
    for (int i = 0; i < 4; ++i)
        if (d->dims[i] < min_dims[i]) return CONV_ERR_BAD_PARAM;
    // order the non-unit dims by stride
    int idx[4], n = 0;
    for (int i = 0; i < 4; ++i) {
        if (d->dims[i] > 1) {
            if (d->strides[i] < 1) return CONV_ERR_BAD_STRIDES;
            idx[n++] = i;
        }
    }
    for (int j = 1; j < n; ++j) {  // insertion sort by stride
        const int v = idx[j];
        int i = j - 1;
        while (i >= 0 && d->strides[idx[i]] > d->strides[v]) {
            idx[i + 1] = idx[i];
            --i;
        }
        idx[i + 1] = v;
    }
    int64_t span = 0;  // largest offset reachable with the dims seen so far
    for (int j = 0; j < n; ++j) {
        int i = idx[j];
        if (d->strides[i] <= span) return CONV_ERR_BAD_STRIDES;  // aliasing
        int64_t t;
        if (!mul_ok(d->dims[i] - 1, d->strides[i], &t)) return CONV_ERR_TOO_LARGE;
        span += t;
        if (span > (INT64_MAX >> 4)) return CONV_ERR_TOO_LARGE;
    }
    for (int i = 0; i < 4; ++i)
        if (d->dims[i] == 0) return CONV_OK;  // empty tensor: nothing is addressed
    int64_t bytes;
    if (!mul_ok(span + 1, elem_size(dtype), &bytes)) return CONV_ERR_TOO_LARGE;
    if ((uint64_t)bytes > d->capacity_bytes) return CONV_ERR_BUFFER_TOO_SMALL;
    return CONV_OK;
}

static int64_t out_extent(int64_t in, int64_t pre, int64_t post, int64_t taps, int64_t dil,
                          int64_t stride) {
    int64_t span = in + pre + post - dil * (taps - 1) - 1;
    if (span < 0) return 0;
    return span / stride + 1;
}

static conv_status check_params(const conv_fprop_params *p) {
    if (!p) return CONV_ERR_NULL_PTR;
    if (p->compute_dtype != CONV_INT32) return CONV_ERR_UNSUPPORTED_COMPUTE;
    for (int i = 0; i < 2; ++i) {
        if (p->stride[i] < 1 || p->dilation[i] < 1) return CONV_ERR_BAD_PARAM;
        if (p->pre_padding[i] < 0 || p->post_padding[i] < 0) return CONV_ERR_BAD_PARAM;
        if (p->stride[i] > (1 << 20) || p->dilation[i] > (1 << 20) || p->pre_padding[i] > (1 << 30) ||
            p->post_padding[i] > (1 << 30))
            return CONV_ERR_TOO_LARGE;
    }
    if (p->mode != CONV_CROSS_CORRELATION && p->mode != CONV_CONVOLUTION) return CONV_ERR_BAD_PARAM;
    if (p->epilogue & ~(CONV_EPILOGUE_BIAS | CONV_EPILOGUE_RELU | CONV_EPILOGUE_INT8_OUT)) return CONV_ERR_BAD_PARAM;
    if (p->out_shift < 0 || p->out_shift > 31 || p->reserved != 0) return CONV_ERR_BAD_PARAM;
    if (p->out_shift != 0 && !(p->epilogue & CONV_EPILOGUE_INT8_OUT)) return CONV_ERR_BAD_PARAM;
    if (p->algo < CONV_ALGO_AUTO || p->algo > CONV_ALGO_IMPLICIT_GEMM_GLOBAL_LOADS) return CONV_ERR_BAD_PARAM;
    return CONV_OK;
}

void make_geom(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
               const conv_fprop_params *p, ConvGeom *g) {
    g->N = x->dims[0]; g->C = x->dims[1]; g->H = x->dims[2]; g->W = x->dims[3];
    g->K = w->dims[0]; g->R = w->dims[2]; g->S = w->dims[3];
    g->P = y->dims[2]; g->Q = y->dims[3];
    for (int i = 0; i < 4; ++i) {
        // a unit dim's stride is never used with a non-zero index; zero it so
        // that kernels may multiply it freely
        g->xs[i] = x->dims[i] > 1 ? x->strides[i] : 0;
        g->ws[i] = w->dims[i] > 1 ? w->strides[i] : 0;
        g->ys[i] = y->dims[i] > 1 ? y->strides[i] : 0;
    }
    g->pad_h = p->pre_padding[0]; g->pad_w = p->pre_padding[1];
    g->str_h = p->stride[0]; g->str_w = p->stride[1];
    g->dil_h = p->dilation[0]; g->dil_w = p->dilation[1];
    g->mode = p->mode;
    g->bias = (p->epilogue & CONV_EPILOGUE_BIAS) != 0;
    g->relu = (p->epilogue & CONV_EPILOGUE_RELU) != 0;
    g->out_int8 = (p->epilogue & CONV_EPILOGUE_INT8_OUT) != 0;
    g->out_shift = p->out_shift;
}

// The gradients take the forward convolution's parameters without an
// epilogue: no bias, ReLU or int8 output, and the algorithm AUTO, IMPLICIT_GEMM
// or DIRECT_GENERIC.
static conv_status check_grad_params(const conv_fprop_params *p) {
    conv_status st = check_params(p);
    if (st) return st;
    if (p->epilogue != 0 || p->out_shift != 0) return CONV_ERR_BAD_PARAM;
    if (p->algo != CONV_ALGO_AUTO && p->algo != CONV_ALGO_IMPLICIT_GEMM && p->algo != CONV_ALGO_DIRECT_GENERIC)
        return CONV_ERR_BAD_PARAM;
    return CONV_OK;
}

// Shapes of a gradient call: image [N,C,H,W], filter [K,C,R,S] and loss
// gradient [N,K,P,Q] with P, Q the forward output size of H, W.  `terms` is
// the largest number of products summed into one result.
static conv_status check_grad_shapes(const conv_tensor_desc *img, const conv_tensor_desc *flt,
                                     const conv_tensor_desc *dy, const conv_fprop_params *p, int64_t terms) {
    if (img->dims[0] != dy->dims[0] || img->dims[1] != flt->dims[1] || flt->dims[0] != dy->dims[1])
        return CONV_ERR_SHAPE_MISMATCH;
    for (int i = 0; i < 2; ++i) {
        const int64_t o = out_extent(img->dims[2 + i], p->pre_padding[i], p->post_padding[i], flt->dims[2 + i],
                                     p->dilation[i], p->stride[i]);
        if (o < 1) return CONV_ERR_BAD_PARAM;
        if (dy->dims[2 + i] != o) return CONV_ERR_SHAPE_MISMATCH;
    }
    if (terms > (int64_t)(INT32_MAX / (128 * 128))) return CONV_ERR_OVERFLOW_RISK;
    int64_t m;
    if (!mul_ok(img->dims[0], img->dims[2], &m) || !mul_ok(m, img->dims[3], &m) || m > (int64_t)INT32_MAX - 256)
        return CONV_ERR_TOO_LARGE;
    if (!mul_ok(dy->dims[0], dy->dims[2], &m) || !mul_ok(m, dy->dims[3], &m) || m > (int64_t)INT32_MAX - 256)
        return CONV_ERR_TOO_LARGE;
    if (flt->dims[0] > (1 << 24) || flt->dims[1] > (1 << 24)) return CONV_ERR_TOO_LARGE;
    return CONV_OK;
}

conv_status validate_dgrad(const conv_tensor_desc *dy, const conv_tensor_desc *w, const conv_tensor_desc *dx,
                           const conv_fprop_params *p) {
    if (!dy || !w || !dx || !p) return CONV_ERR_NULL_PTR;
    conv_status st = check_grad_params(p);
    if (st) return st;
    const int64_t img_min[4] = {0, 1, 1, 1}, flt_min[4] = {1, 1, 1, 1}, dy_min[4] = {0, 1, 1, 1};
    if ((st = check_desc(dy, CONV_INT8, dy_min)) || (st = check_desc(w, CONV_INT8, flt_min)) ||
        (st = check_desc(dx, CONV_INT32, img_min)))
        return st;
    int64_t terms = 0;  // dX sums over k and the taps
    if (!mul_ok(w->dims[0], w->dims[2], &terms) || !mul_ok(terms, w->dims[3], &terms)) return CONV_ERR_OVERFLOW_RISK;
    return check_grad_shapes(dx, w, dy, p, terms);
}

conv_status validate_wgrad(const conv_tensor_desc *x, const conv_tensor_desc *dy, const conv_tensor_desc *dw,
                           const conv_fprop_params *p) {
    if (!x || !dy || !dw || !p) return CONV_ERR_NULL_PTR;
    conv_status st = check_grad_params(p);
    if (st) return st;
    const int64_t img_min[4] = {0, 1, 1, 1}, flt_min[4] = {1, 1, 1, 1}, dy_min[4] = {0, 1, 1, 1};
    if ((st = check_desc(x, CONV_INT8, img_min)) || (st = check_desc(dy, CONV_INT8, dy_min)) ||
        (st = check_desc(dw, CONV_INT32, flt_min)))
        return st;
    int64_t terms = 0;  // dW sums over the batch and the output pixels
    if (!mul_ok(dy->dims[0], dy->dims[2], &terms) || !mul_ok(terms, dy->dims[3], &terms))
        return CONV_ERR_OVERFLOW_RISK;
    return check_grad_shapes(x, dw, dy, p, terms);
}

}  // namespace i8c

using namespace i8c;

extern "C" {

void conv_params_init(conv_fprop_params *p) {
    if (!p) return;
    std::memset(p, 0, sizeof(*p));
    p->stride[0] = p->stride[1] = 1;
    p->dilation[0] = p->dilation[1] = 1;
    p->mode = CONV_CROSS_CORRELATION;
    p->compute_dtype = CONV_INT32;
    p->epilogue = 0;
    p->algo = CONV_ALGO_AUTO;
}

void conv_params_set_symmetric_padding(conv_fprop_params *p, const int64_t pad[2]) {
    if (!p || !pad) return;
    p->pre_padding[0] = p->post_padding[0] = pad[0];
    p->pre_padding[1] = p->post_padding[1] = pad[1];
}

conv_status conv_tensor_desc_packed(conv_tensor_desc *d, int32_t dtype, const int64_t dims[4],
                                    const char *layout) {
    if (!d || !dims || !layout) return CONV_ERR_NULL_PTR;
    if (dtype != CONV_INT8 && dtype != CONV_INT32) return CONV_ERR_DTYPE;
    // memory order, outermost first, as logical dim indices
    int order[4];
    if (!std::strcmp(layout, "NCHW") || !std::strcmp(layout, "KCRS")) {
        int o[4] = {0, 1, 2, 3};
        std::memcpy(order, o, sizeof(o));
    } else if (!std::strcmp(layout, "NHWC") || !std::strcmp(layout, "KRSC")) {
        int o[4] = {0, 2, 3, 1};
        std::memcpy(order, o, sizeof(o));
    } else {
        return CONV_ERR_BAD_PARAM;
    }
    for (int i = 0; i < 4; ++i)
        if (dims[i] < 1) return CONV_ERR_BAD_PARAM;
    d->dtype = dtype;
    d->rank = 4;
    int64_t acc = 1;
    for (int j = 3; j >= 0; --j) {
        int i = order[j];
        d->dims[i] = dims[i];
        d->strides[i] = acc;
        if (!mul_ok(acc, dims[i], &acc)) return CONV_ERR_TOO_LARGE;
    }
    d->capacity_bytes = (uint64_t)acc * (uint64_t)elem_size(dtype);
    return CONV_OK;
}

conv_status conv_fprop_output_dims(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                   const conv_fprop_params *p, int64_t out_dims[4]) {
    if (!x || !w || !p || !out_dims) return CONV_ERR_NULL_PTR;
    if (x->rank != 4 || w->rank != 4) return CONV_ERR_RANK;
    conv_status st = check_params(p);
    if (st) return st;
    if (x->dims[1] != w->dims[1]) return CONV_ERR_SHAPE_MISMATCH;
    for (int i = 1; i < 4; ++i)
        if (x->dims[i] < 1 || w->dims[i] < 1) return CONV_ERR_BAD_PARAM;
    if (x->dims[0] < 0 || w->dims[0] < 0) return CONV_ERR_BAD_PARAM;
    out_dims[0] = x->dims[0];
    out_dims[1] = w->dims[0];
    out_dims[2] = out_extent(x->dims[2], p->pre_padding[0], p->post_padding[0], w->dims[2],
                             p->dilation[0], p->stride[0]);
    out_dims[3] = out_extent(x->dims[3], p->pre_padding[1], p->post_padding[1], w->dims[3],
                             p->dilation[1], p->stride[1]);
    if (out_dims[2] < 1 || out_dims[3] < 1) return CONV_ERR_BAD_PARAM;
    return CONV_OK;
}

conv_status conv_fprop_validate(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                const conv_tensor_desc *y, const conv_fprop_params *p,
                                int64_t bias_elems) {
    if (!x || !w || !y || !p) return CONV_ERR_NULL_PTR;
    conv_status st = check_params(p);
    if (st) return st;
    const int64_t img_min[4] = {0, 1, 1, 1};
    const int64_t flt_min[4] = {0, 1, 1, 1};
    const int64_t out_min[4] = {0, 0, 1, 1};
    if ((st = check_desc(x, CONV_INT8, img_min))) return st;
    if ((st = check_desc(w, CONV_INT8, flt_min))) return st;
    // the output type is what the caller asked for, never a default
    const int32_t y_type = (p->epilogue & CONV_EPILOGUE_INT8_OUT) ? CONV_INT8 : CONV_INT32;
    if ((st = check_desc(y, y_type, out_min))) return st;
    int64_t od[4];
    if ((st = conv_fprop_output_dims(x, w, p, od))) return st;
    for (int i = 0; i < 4; ++i)
        if (y->dims[i] != od[i]) return CONV_ERR_SHAPE_MISMATCH;
    // |acc| <= C*R*S*2^14 must fit int32 so that integer accumulation is exact
    const int64_t crs_max = (int64_t)(INT32_MAX / (128 * 128));
    int64_t crs = 0;
    if (!mul_ok(x->dims[1], w->dims[2], &crs) || !mul_ok(crs, w->dims[3], &crs) || crs > crs_max)
        return CONV_ERR_OVERFLOW_RISK;
    if ((p->epilogue & CONV_EPILOGUE_BIAS) && bias_elems < w->dims[0]) return CONV_ERR_BUFFER_TOO_SMALL;
    // index range of the kernels: pixel and tile counts stay below 2^31
    int64_t m;
    if (!mul_ok(od[0], od[2], &m) || !mul_ok(m, od[3], &m) || m > (int64_t)INT32_MAX - 256)
        return CONV_ERR_TOO_LARGE;
    if (od[1] > (1 << 24) || x->dims[1] > (1 << 24)) return CONV_ERR_TOO_LARGE;
    return CONV_OK;
}

const char *conv_status_string(conv_status s) {
    switch (s) {
        case CONV_OK: return "CONV_OK";
        case CONV_ERR_NULL_PTR: return "CONV_ERR_NULL_PTR: a required pointer is NULL";
        case CONV_ERR_RANK: return "CONV_ERR_RANK: descriptor rank is not 4";
        case CONV_ERR_DTYPE:
            return "CONV_ERR_DTYPE: image/filter must be INT8, output INT32 (INT8 only with CONV_EPILOGUE_INT8_OUT)";
        case CONV_ERR_SHAPE_MISMATCH: return "CONV_ERR_SHAPE_MISMATCH: dims of image, filter and output disagree";
        case CONV_ERR_BAD_STRIDES: return "CONV_ERR_BAD_STRIDES: non-positive or aliasing strides";
        case CONV_ERR_BUFFER_TOO_SMALL: return "CONV_ERR_BUFFER_TOO_SMALL: buffer smaller than the descriptor's extent";
        case CONV_ERR_BAD_PARAM: return "CONV_ERR_BAD_PARAM: bad stride, dilation, padding, mode, flag or empty output";
        case CONV_ERR_OVERFLOW_RISK: return "CONV_ERR_OVERFLOW_RISK: C*R*S*2^14 exceeds int32";
        case CONV_ERR_UNSUPPORTED_COMPUTE: return "CONV_ERR_UNSUPPORTED_COMPUTE: compute type must be INT32";
        case CONV_ERR_ALIGNMENT: return "CONV_ERR_ALIGNMENT: the forced algorithm cannot take these pointers or strides";
        case CONV_ERR_CUDA: return "CONV_ERR_CUDA: a CUDA runtime call failed";
        case CONV_ERR_DEVICE_TIMEOUT: return "CONV_ERR_DEVICE_TIMEOUT: a kernel gave up waiting";
        case CONV_ERR_WORKSPACE: return "CONV_ERR_WORKSPACE: workspace missing or too small";
        case CONV_ERR_UNSUPPORTED_DEVICE: return "CONV_ERR_UNSUPPORTED_DEVICE: current device is not sm_103";
        case CONV_ERR_OVERLAP: return "CONV_ERR_OVERLAP: output overlaps an input or the workspace";
        case CONV_ERR_TOO_LARGE: return "CONV_ERR_TOO_LARGE: extent beyond the library's index range";
        case CONV_ERR_STATIC_WORKSPACE_LIMIT:
            return "CONV_ERR_STATIC_WORKSPACE_LIMIT: the call needs more scratch than the library's static array";
    }
    return "unknown conv_status";
}

int32_t conv_library_version(void) { return 100; }

}  // extern "C"
