// grad.cu -- data and weight gradients of the INT8 convolution (cuDNN
// "Convolutions", sections "Convolution Dgrad" and "Convolution Wgrad"): the
// transposes of the forward sum with respect to the image and to the filter.
//
// dgrad, dX[n,c,h,w] = sum over k, r, s of dY[n,k,p,q] * W[k,c,r',s'] with
// p = (h + pre_h - r*dil_h) / stride_h exact and in range (q likewise):
//  * split by the residues (rho_h, rho_w) of h and w modulo the stride.  The
//    pixels h = rho + i*stride of one residue are reached only by the taps
//    with r*dil = rho + pre (mod stride), r = r0 + t*delta (delta =
//    stride / gcd(dil, stride)), and p = i + c0 - t*e with e = dil*delta /
//    stride and c0 = (rho + pre - r0*dil) / stride.  So each residue class is
//    a stride-1 forward convolution of dY, dilation e, pre-padding
//    (T-1)*e - c0, by the filter's taps r0, r0 + delta, ... taken backwards,
//    K and C exchanged, written into dX through its strides times the stride.
//    With stride 1 there is one class, the whole filter reversed.  Each class
//    runs on the tensor-core kernel with its own filter repack in its own
//    part of the workspace (all repacks in one launch); several classes run
//    side by side on streams forked from the caller's and joined back to it,
//    reading one shared channels-last copy of dY when dY needs one; a class
//    no tap reaches is zero-filled.
//  * otherwise (a class the tensor-core kernel cannot express, more than
//    kMaxDgradPhases classes, or DIRECT_GENERIC): a CUDA-core kernel, one
//    thread per dX element.
// wgrad, dW[k,c,r',s'] = sum over n, p, q of dY[n,k,p,q] * X[n,c,h,w]:
//  * a forward convolution whose image is X with its batch and channel dims
//    exchanged ([C][N][H][W]), whose filter is dY ([K][N][P][Q]: the batch
//    as channels, the output pixels as taps), with the forward stride and
//    dilation exchanged, and whose [C][K][R][S] output is dW with its first
//    two dims exchanged (taps written backwards in CONVOLUTION mode).  Its
//    few output tiles have long reductions (N*P*Q), which the tensor-core
//    kernel cuts into runs over the SMs and adds back up.  With a batch of
//    N <= 32 (N of each k-step's 64 channels), T columns of dY are folded
//    into the channels (channel t*N + n) against a copy of the image T
//    times its size: the same products in T times fewer k-steps.
//  * otherwise (or with DIRECT_GENERIC): a CUDA-core kernel, one warp per dW
//    element, the lanes splitting the n, p, q sum (int32 partial sums, exact
//    by the validator's bound, added across the warp with shuffles).
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <numeric>
#include <vector>

#include "internal.h"

namespace i8c {
namespace {

struct GradArgs {
    const int8_t *a;  // dgrad: dY; wgrad: X
    const int8_t *b;  // dgrad: W;  wgrad: dY
    int32_t *out;     // dgrad: dX; wgrad: dW
    int64_t N, C, H, W, K, R, S, P, Q;
    int64_t xs[4], ws[4], ys[4];  // strides of the image (or dX), the filter (or dW), dY
    int64_t pad_h, pad_w, str_h, str_w, dil_h, dil_w;
    int32_t mode;
};

__global__ void __launch_bounds__(256) dgrad_direct_kernel(const GradArgs g) {
    const int64_t total = g.N * g.C * g.H * g.W;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t w = i % g.W;
        int64_t t = i / g.W;
        const int64_t h = t % g.H;
        t /= g.H;
        const int64_t c = t % g.C;
        const int64_t n = t / g.C;
        int32_t acc = 0;
        for (int64_t r = 0; r < g.R; ++r) {
            const int64_t th = h + g.pad_h - r * g.dil_h;
            if (th < 0 || th % g.str_h) continue;
            const int64_t p = th / g.str_h;
            if (p >= g.P) continue;
            const int64_t rf = g.mode ? g.R - 1 - r : r;
            for (int64_t s = 0; s < g.S; ++s) {
                const int64_t tw = w + g.pad_w - s * g.dil_w;
                if (tw < 0 || tw % g.str_w) continue;
                const int64_t q = tw / g.str_w;
                if (q >= g.Q) continue;
                const int64_t sf = g.mode ? g.S - 1 - s : s;
                const int8_t *dy = g.a + n * g.ys[0] + p * g.ys[2] + q * g.ys[3];
                const int8_t *wk = g.b + c * g.ws[1] + rf * g.ws[2] + sf * g.ws[3];
                for (int64_t k = 0; k < g.K; ++k)
                    acc += (int32_t)__ldg(dy + k * g.ys[1]) * (int32_t)__ldg(wk + k * g.ws[0]);
            }
        }
        g.out[n * g.xs[0] + c * g.xs[1] + h * g.xs[2] + w * g.xs[3]] = acc;
    }
}

__global__ void __launch_bounds__(256) wgrad_direct_kernel(const GradArgs g) {
    const int64_t total = g.K * g.C * g.R * g.S;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t npq = g.N * g.P * g.Q;
    for (int64_t e = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; e < total; e += warps) {
        const int64_t sf = e % g.S;
        int64_t t = e / g.S;
        const int64_t rf = t % g.R;
        t /= g.R;
        const int64_t c = t % g.C;
        const int64_t k = t / g.C;
        // the spatial tap whose products land in filter element (rf, sf)
        const int64_t r = g.mode ? g.R - 1 - rf : rf;
        const int64_t s = g.mode ? g.S - 1 - sf : sf;
        int32_t acc = 0;
        for (int64_t i = lane; i < npq; i += 32) {
            const int64_t q = i % g.Q;
            const int64_t t2 = i / g.Q;
            const int64_t p = t2 % g.P;
            const int64_t n = t2 / g.P;
            const int64_t h = p * g.str_h - g.pad_h + r * g.dil_h;
            const int64_t w = q * g.str_w - g.pad_w + s * g.dil_w;
            if (h < 0 || h >= g.H || w < 0 || w >= g.W) continue;
            acc += (int32_t)__ldg(g.b + n * g.ys[0] + k * g.ys[1] + p * g.ys[2] + q * g.ys[3]) *
                   (int32_t)__ldg(g.a + n * g.xs[0] + c * g.xs[1] + h * g.xs[2] + w * g.xs[3]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) g.out[k * g.ws[0] + c * g.ws[1] + rf * g.ws[2] + sf * g.ws[3]] = acc;
    }
}

// Strides of a descriptor with those of unit dims zeroed (never multiplied by
// a non-zero index).
void unit_strides(const conv_tensor_desc *d, int64_t out[4]) {
    for (int i = 0; i < 4; ++i) out[i] = d->dims[i] > 1 ? d->strides[i] : 0;
}

GradArgs grad_args(const conv_tensor_desc *img, const conv_tensor_desc *flt, const conv_tensor_desc *dy,
                   const conv_fprop_params *p) {
    GradArgs g;
    g.N = img->dims[0]; g.C = img->dims[1]; g.H = img->dims[2]; g.W = img->dims[3];
    g.K = flt->dims[0]; g.R = flt->dims[2]; g.S = flt->dims[3];
    g.P = dy->dims[2]; g.Q = dy->dims[3];
    unit_strides(img, g.xs);
    unit_strides(flt, g.ws);
    unit_strides(dy, g.ys);
    g.pad_h = p->pre_padding[0]; g.pad_w = p->pre_padding[1];
    g.str_h = p->stride[0]; g.str_w = p->stride[1];
    g.dil_h = p->dilation[0]; g.dil_w = p->dilation[1];
    g.mode = p->mode;
    return g;
}

int grid_for(int64_t items, int per_block) {
    int64_t blocks = (items + per_block - 1) / per_block;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    return (int)(blocks < 1 ? 1 : blocks);
}

// More residue classes than this (stride_h * stride_w) take the CUDA-core
// kernel: each class costs a filter repack and a launch.
constexpr int64_t kMaxDgradPhases = 64;

__global__ void __launch_bounds__(256) zero_view_kernel(int32_t *y, int64_t N, int64_t C, int64_t P, int64_t Q,
                                                        int64_t s0, int64_t s1, int64_t s2, int64_t s3) {
    const int64_t total = N * C * P * Q;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = i % Q, t = i / Q, p = t % P, t2 = t / P, c = t2 % C, n = t2 / C;
        y[n * s0 + c * s1 + p * s2 + q * s3] = 0;
    }
}

// One residue class (rho_h, rho_w) of dX's pixels under the stride, as a
// forward convolution of dY (see the top of the file).
struct DgradPhase {
    ConvGeom g;        // image dY, filter the class's taps, output the class's dX pixels
    IgemmPlan pl;
    int64_t w_origin;  // element offset in W of the class filter's tap (0, 0)
    int64_t y_origin;  // element offset in dX of the class's first pixel
    size_t ws_off;     // the class's own part of the workspace
    bool taps;         // false: no tap reaches the class, its pixels are zero
};

// Streams the residue classes of one dgrad call run on side by side, forked
// from the caller's stream and joined back to it, with the events that fork
// and join them; created on first use, one set per device, kept for the life
// of the process.  One call at a time uses a set (its mutex), so that two
// host threads never record the same event between the other's record and
// wait.
constexpr int kSideStreams = 4;
constexpr int kSideDevices = 64;

struct SideSet {
    std::mutex mu;
    cudaStream_t streams[kSideStreams] = {};
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[kSideStreams] = {};
    bool ready = false;
};

SideSet *side_set() {
    static std::mutex mu;
    static SideSet sets[kSideDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSideDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    SideSet &ss = sets[dev];
    if (!ss.ready) {
        bool ok = ss.fork || cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < kSideStreams && ok; ++i) {
            ok = ss.streams[i] || cudaStreamCreateWithFlags(&ss.streams[i], cudaStreamNonBlocking) == cudaSuccess;
            ok = ok && (ss.join[i] || cudaEventCreateWithFlags(&ss.join[i], cudaEventDisableTiming) == cudaSuccess);
        }
        if (!ok) return nullptr;  // what was created stays for the next try
        ss.ready = true;
    }
    return &ss;
}

// The taps of one axis that reach residue rho: r = r0 + t*delta, t < T.
// Returns T (0 when none), with r0, delta, the class's dilation e and its
// pre-padding.
int64_t phase_axis(int64_t rho, int64_t pre, int64_t str, int64_t dil, int64_t taps, int64_t *r0, int64_t *delta,
                   int64_t *e, int64_t *pad) {
    const int64_t gcd = std::gcd(dil, str);
    *delta = str / gcd;
    *e = dil / gcd;
    // r*dil = rho + pre (mod str) has its solutions every delta taps, the
    // first below delta when there are any
    for (int64_t r = 0; r < *delta && r < taps; ++r) {
        if ((r * dil - rho - pre) % str != 0) continue;
        const int64_t T = (taps - r + *delta - 1) / *delta;
        const int64_t c0 = (rho + pre - r * dil) / str;  // exact
        *r0 = r;
        *pad = (T - 1) * *e - c0;
        return T;
    }
    return 0;
}

// dgrad as stride_h * stride_w forward convolutions of dY, one per residue
// class; returns false when the tensor-core kernel cannot take one of them.
bool dgrad_phases(const conv_tensor_desc *dy, const conv_tensor_desc *w, const conv_tensor_desc *dx,
                  const conv_fprop_params *p, std::vector<DgradPhase> *out) {
    const int64_t sh = p->stride[0], sw = p->stride[1];
    if (sh * sw > kMaxDgradPhases) return false;
    int64_t ys[4], fs[4], xs[4];
    unit_strides(dy, ys);
    unit_strides(w, fs);
    unit_strides(dx, xs);
    const int64_t R = w->dims[2], S = w->dims[3], H = dx->dims[2], W = dx->dims[3];
    for (int64_t rh = 0; rh < sh && rh < H; ++rh) {
        for (int64_t rw = 0; rw < sw && rw < W; ++rw) {
            DgradPhase ph = {};
            ConvGeom &g = ph.g;
            // output: the class's pixels of dX, [N][C][P'][Q']
            g.N = dy->dims[0];
            g.K = dx->dims[1];
            g.P = (H - rh + sh - 1) / sh;
            g.Q = (W - rw + sw - 1) / sw;
            g.ys[0] = xs[0]; g.ys[1] = xs[1]; g.ys[2] = sh * xs[2]; g.ys[3] = sw * xs[3];
            ph.y_origin = rh * xs[2] + rw * xs[3];
            int64_t r0 = 0, dh = 1, eh = 1, padh = 0, s0 = 0, dw = 1, ew = 1, padw = 0;
            const int64_t th = phase_axis(rh, p->pre_padding[0], sh, p->dilation[0], R, &r0, &dh, &eh, &padh);
            const int64_t tw = phase_axis(rw, p->pre_padding[1], sw, p->dilation[1], S, &s0, &dw, &ew, &padw);
            ph.taps = th > 0 && tw > 0 && dy->dims[1] > 0;
            if (ph.taps) {
                // image: dY, its K channels the reduction
                g.C = dy->dims[1]; g.H = dy->dims[2]; g.W = dy->dims[3];
                for (int i = 0; i < 4; ++i) g.xs[i] = ys[i];
                // filter [C][K][T_h][T_w]: tap (u, v) is r = r0 + (T_h-1-u)*delta_h
                // (s likewise), stored at r' = r or R-1-r by the mode
                g.R = th; g.S = tw;
                g.ws[0] = fs[1];
                g.ws[1] = fs[0];
                const int64_t rl = r0 + (th - 1) * dh, sl = s0 + (tw - 1) * dw;  // the taps of u, v = 0
                if (p->mode == CONV_CONVOLUTION) {
                    ph.w_origin = (R - 1 - rl) * fs[2] + (S - 1 - sl) * fs[3];
                    g.ws[2] = dh * fs[2];
                    g.ws[3] = dw * fs[3];
                } else {
                    ph.w_origin = rl * fs[2] + sl * fs[3];
                    g.ws[2] = -dh * fs[2];
                    g.ws[3] = -dw * fs[3];
                }
                g.pad_h = padh; g.pad_w = padw;
                g.str_h = g.str_w = 1;
                g.dil_h = eh; g.dil_w = ew;
                g.mode = CONV_CROSS_CORRELATION;
                g.bias = g.relu = g.out_int8 = false;
                g.out_shift = 0;
                if (!igemm_supported(g)) return false;
            }
            out->push_back(ph);
        }
    }
    return true;
}

// wgrad as a forward convolution (see the top of the file); fills g and the
// element offset of the output's origin (non-zero when CONVOLUTION mode runs
// the output taps backwards) and returns true when the tensor-core kernel
// takes it.
bool wgrad_as_fprop(const conv_tensor_desc *x, const conv_tensor_desc *dy, const conv_tensor_desc *dw,
                    const conv_fprop_params *p, ConvGeom *g, int64_t *y_origin) {
    int64_t xs[4], ys[4], ds[4];
    unit_strides(x, xs);
    unit_strides(dy, ys);
    unit_strides(dw, ds);
    // image: the batch becomes the channels, the channels the batch
    g->N = x->dims[1]; g->C = x->dims[0]; g->H = x->dims[2]; g->W = x->dims[3];
    g->xs[0] = xs[1]; g->xs[1] = xs[0]; g->xs[2] = xs[2]; g->xs[3] = xs[3];
    // filter: dY, its batch as channels, its P x Q pixels as taps
    g->K = dy->dims[1]; g->R = dy->dims[2]; g->S = dy->dims[3];
    g->ws[0] = ys[1]; g->ws[1] = ys[0]; g->ws[2] = ys[2]; g->ws[3] = ys[3];
    // output [C][K][R][S]: dW with its first two dims exchanged
    g->P = dw->dims[2]; g->Q = dw->dims[3];
    g->ys[0] = ds[1]; g->ys[1] = ds[0]; g->ys[2] = ds[2]; g->ys[3] = ds[3];
    *y_origin = 0;
    if (p->mode == CONV_CONVOLUTION) {  // dW[k,c,R-1-r,S-1-s] holds tap (r, s)
        *y_origin = (g->P - 1) * ds[2] + (g->Q - 1) * ds[3];
        g->ys[2] = -ds[2];
        g->ys[3] = -ds[3];
    }
    // h = r*dil - pre + p*stride: the forward stride and dilation change places
    g->pad_h = p->pre_padding[0]; g->pad_w = p->pre_padding[1];
    g->str_h = p->dilation[0]; g->str_w = p->dilation[1];
    g->dil_h = p->stride[0]; g->dil_w = p->stride[1];
    g->mode = CONV_CROSS_CORRELATION;
    g->bias = g->relu = g->out_int8 = false;
    g->out_shift = 0;
    if (!igemm_supported(*g)) return false;
    // the repacked loss gradient grows with P*Q*ceil(N/64) f16 blocks: keep it
    // within a few GB
    const int64_t blocks = ((g->K + 255) / 256) * g->R * g->S * ((g->C + 63) / 64);
    return blocks * 256 * 128 <= ((int64_t)4 << 30);
}

// The folded weight gradient (see WgradFold): with a batch of N <= 32 the
// forward convolution above fills only N of each k-step's 64 channels.
// Folding T = min(64 / N, Q, 8) output columns of dY into the channels
// (channel t*N + n) turns the Q taps along W into Q2 = ceil(Q / T), read
// from a copy X'' of the image in which channel t*N + n of column u is
// X[n, c, h, u - pre_w + t*stride_w]: the same products, T times fewer
// k-steps, for a copy T times the image.  Along W the folded convolution has
// no padding (X'' starts at the padded origin), the tap q2 at dilation
// T*stride_w and the output column s at stride dilation_w; along H it is
// the convolution above.  Returns false (no folding) where it does not
// apply or does not fit.
bool wgrad_fold(const conv_tensor_desc *x, const conv_tensor_desc *dy, const conv_fprop_params *p,
                const ConvGeom &g, ConvGeom *g2, WgradFold *f) {
    const int64_t N = x->dims[0], Q = dy->dims[3];
    if (N < 1 || N > 32) return false;
    int64_t T = 64 / N;
    if (T > Q) T = Q;
    if (T > 8) T = 8;
    if (T < 2) return false;
    std::memset(f, 0, sizeof(*f));
    unit_strides(x, f->xs);
    unit_strides(dy, f->ys);
    f->N = N; f->C = x->dims[1]; f->H = x->dims[2]; f->W = x->dims[3];
    f->K = dy->dims[1]; f->P = dy->dims[2]; f->Q = Q;
    f->T = T;
    f->Q2 = (Q + T - 1) / T;
    f->c16 = (T * N + 15) / 16 * 16;
    f->pre_w = p->pre_padding[1];
    f->stride_w = p->stride[1];
    const int64_t S = g.Q;  // dW's columns: the forward convolution's output columns
    f->U = T * f->stride_w * (f->Q2 - 1) + p->dilation[1] * (S - 1) + 1;
    if (f->U >= ((int64_t)1 << 30) || f->C * f->H * f->U * f->c16 > ((int64_t)4 << 30)) return false;
    *g2 = g;
    g2->C = f->c16;
    g2->W = f->U;
    g2->xs[0] = f->H * f->U * f->c16; g2->xs[1] = 1; g2->xs[2] = f->U * f->c16; g2->xs[3] = f->c16;
    g2->S = f->Q2;
    g2->ws[0] = f->P * f->Q2 * f->c16; g2->ws[1] = 1; g2->ws[2] = f->Q2 * f->c16; g2->ws[3] = f->c16;
    g2->pad_w = 0;
    g2->dil_w = T * f->stride_w;
    return igemm_supported(*g2);
}

conv_status plan_wgrad(const conv_tensor_desc *x, const void *x_dev, const conv_tensor_desc *dy,
                       const conv_tensor_desc *dw, const conv_fprop_params *p, ConvGeom *g, int64_t *y_origin,
                       bool *tensor, IgemmPlan *pl, WgradFold *fold, size_t *ws_bytes) {
    conv_status st = validate_wgrad(x, dy, dw, p);
    if (st) return st;
    *tensor = p->algo != CONV_ALGO_DIRECT_GENERIC && wgrad_as_fprop(x, dy, dw, p, g, y_origin);
    if (p->algo == CONV_ALGO_IMPLICIT_GEMM && !*tensor) return CONV_ERR_ALIGNMENT;
    fold->T = 1;
    *ws_bytes = 0;
    if (!*tensor) return CONV_OK;
    ConvGeom g2;
    WgradFold f;
    if (wgrad_fold(x, dy, p, *g, &g2, &f)) {
        IgemmPlan pl2;
        igemm_plan(g2, nullptr, &pl2);
        // the copy is read in place (channels-last, 16-byte aligned) with one
        // channel step per tap
        if (!pl2.pack_x && !pl2.nchw_rows && !pl2.register_loads && pl2.c_steps == 1) {
            *g = g2;
            *pl = pl2;
            *fold = f;
            *ws_bytes = ((pl2.workspace_bytes + 255) & ~(size_t)255) +
                        (size_t)(f.C * f.H * f.U * f.c16);
            return CONV_OK;
        }
    }
    igemm_plan(*g, x_dev, pl);
    *ws_bytes = pl->workspace_bytes;
    return CONV_OK;
}

// Plans a dgrad call: *tensor tells whether the residue classes in *ph run on
// the tensor cores, *ws_bytes the workspace they need (each class its own
// part, so that they can run at the same time).
conv_status plan_dgrad(const conv_tensor_desc *dy, const int8_t *dy_dev, const conv_tensor_desc *w,
                       const conv_tensor_desc *dx, const conv_fprop_params *p, std::vector<DgradPhase> *ph,
                       bool *tensor, size_t *ws_bytes) {
    conv_status st = validate_dgrad(dy, w, dx, p);
    if (st) return st;
    *tensor = p->algo != CONV_ALGO_DIRECT_GENERIC && dgrad_phases(dy, w, dx, p, ph);
    if (p->algo == CONV_ALGO_IMPLICIT_GEMM && !*tensor) return CONV_ERR_ALIGNMENT;
    *ws_bytes = 0;
    if (!*tensor) return CONV_OK;
    int tapped = 0;
    bool pack = false;
    // a class whose window starts inside dY (negative padding) gathers
    // with register loads, which bounds-check every pixel
    auto neg_pad = [](const DgradPhase &c) { return c.g.pad_h < 0 || c.g.pad_w < 0; };
    bool in_place = false;
    for (DgradPhase &c : *ph) {
        if (!c.taps) continue;
        igemm_plan(c.g, dy_dev, &c.pl, neg_pad(c));
        ++tapped;
        pack = pack || c.pl.pack_x;
        in_place = in_place || c.pl.nchw_rows;
    }
    // an NCHW dY is either read in place by every class or copied once for
    // all of them
    if (pack && in_place)
        for (DgradPhase &c : *ph)
            if (c.taps && c.pl.nchw_rows) igemm_plan(c.g, dy_dev, &c.pl, neg_pad(c), false);
    // Every class reads the same dY at stride 1 (every row): when dY needs a
    // channels-last copy, one copy after the classes' parts serves them all,
    // made once before they fork (each part then ends before its own copy).
    const bool share = tapped > 1 && pack;
    for (DgradPhase &c : *ph) {
        if (!c.taps) continue;
        c.ws_off = *ws_bytes;
        const size_t part = share ? c.pl.xpack_off : c.pl.workspace_bytes;
        if (c.g.N > 0) *ws_bytes += (part + 255) & ~(size_t)255;
    }
    if (share) {
        const size_t shared_off = *ws_bytes;
        size_t xbytes = 0;
        for (DgradPhase &c : *ph) {
            if (!c.taps) continue;
            xbytes = c.pl.xpack_bytes;
            c.pl.xpack_off = shared_off - c.ws_off;
            c.pl.workspace_bytes = c.pl.xpack_off + c.pl.xpack_bytes;
            c.pl.pack_done = true;
        }
        *ws_bytes += (xbytes + 255) & ~(size_t)255;
    }
    return CONV_OK;
}

// Plans of recent dgrad calls (residue classes with their plans), keyed like
// forward plans on the descriptors, parameters, device and dY alignment; the
// least recently used give way; conv_shutdown empties it.
constexpr int kDgradCacheSize = 16;
struct DgradCacheEntry {
    PlanKey key;
    std::vector<DgradPhase> ph;
    bool tensor;
    size_t ws;
    uint64_t used;
    bool valid;
};
std::mutex g_dgrad_mu;
DgradCacheEntry g_dgrad_cache[kDgradCacheSize];
uint64_t g_dgrad_clock = 0;

conv_status plan_dgrad_cached(const conv_tensor_desc *dy, const int8_t *dy_dev, const conv_tensor_desc *w,
                              const conv_tensor_desc *dx, const conv_fprop_params *p, std::vector<DgradPhase> *ph,
                              bool *tensor, size_t *ws_bytes) {
    if (!dy || !w || !dx || !p) return CONV_ERR_NULL_PTR;
    int dev = 0;
    cudaGetDevice(&dev);
    const PlanKey key = make_plan_key(dy, w, dx, p, dy_dev, dev);
    {
        std::lock_guard<std::mutex> lock(g_dgrad_mu);
        for (auto &e : g_dgrad_cache)
            if (e.valid && e.key.n == key.n && std::memcmp(e.key.v, key.v, sizeof(int64_t) * key.n) == 0) {
                e.used = ++g_dgrad_clock;
                *ph = e.ph;
                *tensor = e.tensor;
                *ws_bytes = e.ws;
                return CONV_OK;
            }
    }
    conv_status st = plan_dgrad(dy, dy_dev, w, dx, p, ph, tensor, ws_bytes);
    if (st) return st;  // only valid plans are kept
    std::lock_guard<std::mutex> lock(g_dgrad_mu);
    DgradCacheEntry *victim = &g_dgrad_cache[0];
    for (auto &e : g_dgrad_cache) {
        if (!e.valid) {
            victim = &e;
            break;
        }
        if (e.used < victim->used) victim = &e;
    }
    victim->key = key;
    victim->ph = *ph;
    victim->tensor = *tensor;
    victim->ws = *ws_bytes;
    victim->used = ++g_dgrad_clock;
    victim->valid = true;
    return CONV_OK;
}

}  // namespace

void dgrad_cache_clear() {
    std::lock_guard<std::mutex> lock(g_dgrad_mu);
    for (auto &e : g_dgrad_cache) {
        e.valid = false;
        e.ph.clear();
    }
}

}  // namespace i8c

using namespace i8c;

extern "C" {

conv_status conv_dgrad_workspace_size(const conv_tensor_desc *dy, const conv_tensor_desc *w,
                                      const conv_tensor_desc *dx, const conv_fprop_params *p, size_t *bytes) {
    if (!bytes) return CONV_ERR_NULL_PTR;
    std::vector<DgradPhase> ph;
    bool tensor = false;
    size_t ws = 0;
    conv_status st = plan_dgrad_cached(dy, nullptr, w, dx, p, &ph, &tensor, &ws);
    if (st) return st;
    *bytes = ws;
    return CONV_OK;
}

conv_status conv_dgrad(const conv_tensor_desc *dy, const int8_t *dy_dev, const conv_tensor_desc *w,
                       const int8_t *w_dev, const conv_tensor_desc *dx, int32_t *dx_dev,
                       const conv_fprop_params *p, void *workspace, size_t workspace_bytes, void *stream) {
    std::vector<DgradPhase> ph;
    bool tensor = false;
    size_t ws = 0;
    conv_status st = plan_dgrad_cached(dy, dy_dev, w, dx, p, &ph, &tensor, &ws);
    if (st) return st;
    if (dx->dims[0] == 0) return CONV_OK;
    if (!dy_dev || !w_dev || !dx_dev) return CONV_ERR_NULL_PTR;
    const uint64_t dx_bytes = (uint64_t)desc_extent_elems(dx) * 4;
    if (overlaps(dx_dev, dx_bytes, dy_dev, (uint64_t)desc_extent_elems(dy)) ||
        overlaps(dx_dev, dx_bytes, w_dev, (uint64_t)desc_extent_elems(w)) ||
        overlaps(dx_dev, dx_bytes, workspace, workspace_bytes))
        return CONV_ERR_OVERLAP;
    if ((st = check_device())) return st;
    cudaStream_t s = (cudaStream_t)stream;
    if (tensor) {
        if (ws > 0) {
            if (!workspace || workspace_bytes < ws || ((uintptr_t)workspace % 256) != 0) return CONV_ERR_WORKSPACE;
            if (overlaps(workspace, ws, dy_dev, (uint64_t)desc_extent_elems(dy)) ||
                overlaps(workspace, ws, w_dev, (uint64_t)desc_extent_elems(w)))
                return CONV_ERR_OVERLAP;
        }
        // one class: on the caller's stream.  Several: the filters of all
        // classes are repacked on the caller's stream (one launch per
        // kMaxPackJobs classes, each into its own part of the workspace),
        // then each class runs on a side stream forked from the caller's (an
        // event), writing its own dX pixels, and the side streams are joined
        // back (an event each)
        auto run_class = [&](const DgradPhase &c, cudaStream_t cs, bool packed) -> conv_status {
            int32_t *y = dx_dev + c.y_origin;
            if (!c.taps) {
                const ConvGeom &g = c.g;
                zero_view_kernel<<<grid_for(g.N * g.K * g.P * g.Q, 256), 256, 0, cs>>>(
                    y, g.N, g.K, g.P, g.Q, g.ys[0], g.ys[1], g.ys[2], g.ys[3]);
                return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
            }
            void *cw = static_cast<uint8_t *>(workspace) + c.ws_off;
            return igemm_main_launch(c.g, c.pl, dy_dev, w_dev + c.w_origin, y, nullptr, cw, cs, !packed);
        };
        if (ph.empty()) return CONV_OK;
        if (ph.size() == 1) return run_class(ph[0], s, false);
        SideSet *ss = side_set();
        if (!ss) return CONV_ERR_CUDA;
        std::lock_guard<std::mutex> lock(ss->mu);
        // the shared channels-last copy of dY, once
        for (const DgradPhase &c : ph)
            if (c.taps && c.pl.pack_done) {
                if ((st = igemm_pack_image_launch(c.g, c.pl, dy_dev, static_cast<uint8_t *>(workspace) + c.ws_off, s)))
                    return st;
                break;
            }
        {
            const ConvGeom *gs[kMaxPackJobs];
            const IgemmPlan *ps[kMaxPackJobs];
            const int8_t *ws_[kMaxPackJobs];
            void *wk[kMaxPackJobs];
            int n = 0;
            for (size_t i = 0; i <= ph.size(); ++i) {
                if (n == kMaxPackJobs || (i == ph.size() && n > 0)) {
                    if ((st = igemm_pack_filter_group_launch(n, gs, ps, ws_, wk, s))) return st;
                    n = 0;
                }
                if (i == ph.size() || !ph[i].taps) continue;
                gs[n] = &ph[i].g;
                ps[n] = &ph[i].pl;
                ws_[n] = w_dev + ph[i].w_origin;
                wk[n] = static_cast<uint8_t *>(workspace) + ph[i].ws_off;
                ++n;
            }
        }
        // the classes as one launch on the caller's stream when they share a
        // kernel variant and cut no tiles (no fork or join then); the classes
        // no tap reaches are zero-filled beside it
        {
            const ConvGeom *gs[kIgemmMaxGroup];
            const IgemmPlan *ps[kIgemmMaxGroup];
            void *ys[kIgemmMaxGroup];
            void *wk[kIgemmMaxGroup];
            int n = 0;
            bool fits = true;
            for (const DgradPhase &c : ph) {
                if (!c.taps) continue;
                if (n == kIgemmMaxGroup) {
                    fits = false;
                    break;
                }
                gs[n] = &c.g;
                ps[n] = &c.pl;
                ys[n] = dx_dev + c.y_origin;
                wk[n] = static_cast<uint8_t *>(workspace) + c.ws_off;
                ++n;
            }
            bool launched = false;
            // (right behind the repack launch above on the caller's stream)
            if (fits && n >= 2 && (st = igemm_group_launch(n, gs, ps, dy_dev, ys, wk, s, &launched, true))) return st;
            if (launched) {
                for (const DgradPhase &c : ph)
                    if (!c.taps && (st = run_class(c, s, true))) return st;
                return CONV_OK;
            }
        }
        const int nside = (int)ph.size() < kSideStreams ? (int)ph.size() : kSideStreams;
        conv_status rc = cudaEventRecord(ss->fork, s) == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
        for (int i = 0; i < nside && rc == CONV_OK; ++i)
            if (cudaStreamWaitEvent(ss->streams[i], ss->fork, 0) != cudaSuccess) rc = CONV_ERR_CUDA;
        for (size_t i = 0; i < ph.size() && rc == CONV_OK; ++i) rc = run_class(ph[i], ss->streams[i % nside], true);
        // join every side stream back, whatever happened above, so that the
        // caller's stream (or its capture) is left whole
        for (int i = 0; i < nside; ++i)
            if (cudaEventRecord(ss->join[i], ss->streams[i]) != cudaSuccess ||
                cudaStreamWaitEvent(s, ss->join[i], 0) != cudaSuccess)
                rc = CONV_ERR_CUDA;
        return rc;
    }
    const GradArgs a = [&] {
        GradArgs r = grad_args(dx, w, dy, p);
        r.a = dy_dev;
        r.b = w_dev;
        r.out = dx_dev;
        return r;
    }();
    dgrad_direct_kernel<<<grid_for(a.N * a.C * a.H * a.W, 256), 256, 0, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

conv_status conv_wgrad_workspace_size(const conv_tensor_desc *x, const conv_tensor_desc *dy,
                                      const conv_tensor_desc *dw, const conv_fprop_params *p, size_t *bytes) {
    if (!bytes) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    WgradFold fold;
    size_t need = 0;
    int64_t origin = 0;
    bool tensor = false;
    conv_status st = plan_wgrad(x, nullptr, dy, dw, p, &g, &origin, &tensor, &pl, &fold, &need);
    if (st) return st;
    *bytes = (tensor && g.N > 0 && g.K > 0) ? need : 0;
    return CONV_OK;
}

conv_status conv_wgrad(const conv_tensor_desc *x, const int8_t *x_dev, const conv_tensor_desc *dy,
                       const int8_t *dy_dev, const conv_tensor_desc *dw, int32_t *dw_dev,
                       const conv_fprop_params *p, void *workspace, size_t workspace_bytes, void *stream) {
    ConvGeom g;
    IgemmPlan pl;
    WgradFold fold;
    size_t need = 0;
    int64_t origin = 0;
    bool tensor = false;
    conv_status st = plan_wgrad(x, x_dev, dy, dw, p, &g, &origin, &tensor, &pl, &fold, &need);
    if (st) return st;
    // an empty batch reads neither input: only the gradient must be given
    const bool empty_batch = x->dims[0] == 0;
    if (!dw_dev || (!empty_batch && (!x_dev || !dy_dev))) return CONV_ERR_NULL_PTR;
    const uint64_t dw_bytes = (uint64_t)desc_extent_elems(dw) * 4;
    if (overlaps(dw_dev, dw_bytes, x_dev, (uint64_t)desc_extent_elems(x)) ||
        overlaps(dw_dev, dw_bytes, dy_dev, (uint64_t)desc_extent_elems(dy)) ||
        overlaps(dw_dev, dw_bytes, workspace, workspace_bytes))
        return CONV_ERR_OVERLAP;
    if ((st = check_device())) return st;
    // an empty batch gives an all-zero gradient (the CUDA-core kernel writes it)
    if (tensor && x->dims[0] > 0) {
        if (!workspace || workspace_bytes < need || ((uintptr_t)workspace % 256) != 0) return CONV_ERR_WORKSPACE;
        if (overlaps(workspace, need, x_dev, (uint64_t)desc_extent_elems(x)) ||
            overlaps(workspace, need, dy_dev, (uint64_t)desc_extent_elems(dy)))
            return CONV_ERR_OVERLAP;
        if (fold.T > 1) {
            // the copy X'' after the folded convolution's own workspace; the
            // convolution reads the filter blocks the fold repacked
            int8_t *x2 = static_cast<int8_t *>(workspace) + ((pl.workspace_bytes + 255) & ~(size_t)255);
            fold.x = x_dev;
            fold.dy = dy_dev;
            if ((st = igemm_wgrad_fold_launch(fold, pl, x2, workspace, stream))) return st;
            return igemm_main_launch(g, pl, x2, nullptr, dw_dev + origin, nullptr, workspace, stream, false);
        }
        return igemm_main_launch(g, pl, x_dev, dy_dev, dw_dev + origin, nullptr, workspace, stream, true);
    }
    GradArgs a = grad_args(x, dw, dy, p);
    a.a = x_dev;
    a.b = dy_dev;
    a.out = dw_dev;
    wgrad_direct_kernel<<<grid_for(a.K * a.C * a.R * a.S * 32, 256), 256, 0, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // extern "C"
