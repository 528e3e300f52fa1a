// direct.cu -- CUDA-core direct convolution kernels.
//
// Two kernels that take any validated descriptor:
//  * generic: one thread per output element, scalar int32 multiply-adds over
//    (c, r, s), every address from the descriptors' strides.  It is the
//    always-correct path for layouts the tensor-core kernel cannot load.
//  * dp4a: for small channel counts (the forum thread's 1x1x5x5 image and the
//    blog post's 3-channel image).  The reduction index (c, r, s) is flattened
//    and consumed four elements at a time with __dp4a; the filter block and a
//    per-reduction-element offset table live in shared memory, and every
//    thread produces one pixel for kDp4aKB output channels.
// Integer accumulation in int32 is exact: the validator bounds C*R*S*2^14 by
// 2^31-1.  Bias is added with int32 wrap-around, then ReLU.
#include <cuda_runtime.h>

#include "internal.h"

namespace i8c {

struct DirectArgs {
    const int8_t *x;
    const int8_t *w;
    void *y;  // int32 elements, or int8 when out_int8
    const int32_t *bias;
    int64_t N, C, H, W, K, R, S, P, Q;
    int64_t xs0, xs1, xs2, xs3;
    int64_t ws0, ws1, ws2, ws3;
    int64_t ys0, ys1, ys2, ys3;
    int64_t pad_h, pad_w, str_h, str_w, dil_h, dil_w;
    int32_t mode, relu;
    int32_t out_int8, out_shift;
};

static DirectArgs make_args(const ConvGeom &g, const int8_t *x, const int8_t *w, void *y,
                            const int32_t *bias) {
    DirectArgs a;
    a.x = x; a.w = w; a.y = y; a.bias = g.bias ? bias : nullptr;
    a.out_int8 = g.out_int8 ? 1 : 0;
    a.out_shift = g.out_shift;
    a.N = g.N; a.C = g.C; a.H = g.H; a.W = g.W; a.K = g.K; a.R = g.R; a.S = g.S;
    a.P = g.P; a.Q = g.Q;
    a.xs0 = g.xs[0]; a.xs1 = g.xs[1]; a.xs2 = g.xs[2]; a.xs3 = g.xs[3];
    a.ws0 = g.ws[0]; a.ws1 = g.ws[1]; a.ws2 = g.ws[2]; a.ws3 = g.ws[3];
    a.ys0 = g.ys[0]; a.ys1 = g.ys[1]; a.ys2 = g.ys[2]; a.ys3 = g.ys[3];
    a.pad_h = g.pad_h; a.pad_w = g.pad_w; a.str_h = g.str_h; a.str_w = g.str_w;
    a.dil_h = g.dil_h; a.dil_w = g.dil_w;
    a.mode = g.mode; a.relu = g.relu ? 1 : 0;
    return a;
}

__device__ __forceinline__ int32_t finish(int32_t acc, const int32_t *bias, int64_t k, int relu) {
    if (bias) acc = (int32_t)((uint32_t)acc + (uint32_t)__ldg(bias + k));
    if (relu) acc = max(acc, 0);
    return acc;
}

__device__ __forceinline__ void store_out(const DirectArgs &a, int64_t off, int32_t v) {
    if (a.out_int8)
        static_cast<int8_t *>(a.y)[off] = requant_i8(v, a.out_shift);
    else
        static_cast<int32_t *>(a.y)[off] = v;
}

// ---------------------------------------------------------------- generic
__global__ void __launch_bounds__(256) conv_direct_generic_kernel(const DirectArgs a) {
    const int64_t total = a.N * a.K * a.P * a.Q;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        // q fastest so that consecutive threads read neighbouring pixels
        int64_t q = i % a.Q;
        int64_t t = i / a.Q;
        int64_t p = t % a.P;
        t /= a.P;
        int64_t k = t % a.K;
        int64_t n = t / a.K;
        const int64_t h0 = p * a.str_h - a.pad_h;
        const int64_t w0 = q * a.str_w - a.pad_w;
        const int8_t *xn = a.x + n * a.xs0;
        const int8_t *wk = a.w + k * a.ws0;
        int32_t acc = 0;
        for (int64_t r = 0; r < a.R; ++r) {
            const int64_t h = h0 + r * a.dil_h;
            if (h < 0 || h >= a.H) continue;
            const int64_t rf = a.mode ? a.R - 1 - r : r;
            for (int64_t s = 0; s < a.S; ++s) {
                const int64_t w = w0 + s * a.dil_w;
                if (w < 0 || w >= a.W) continue;
                const int64_t sf = a.mode ? a.S - 1 - s : s;
                const int8_t *xp = xn + h * a.xs2 + w * a.xs3;
                const int8_t *wp = wk + rf * a.ws2 + sf * a.ws3;
                for (int64_t c = 0; c < a.C; ++c)
                    acc += (int32_t)__ldg(xp + c * a.xs1) * (int32_t)__ldg(wp + c * a.ws1);
            }
        }
        store_out(a, n * a.ys0 + k * a.ys1 + p * a.ys2 + q * a.ys3, finish(acc, a.bias, k, a.relu));
    }
}

conv_status generic_launch(const ConvGeom &g, const int8_t *x, const int8_t *w, void *y,
                           const int32_t *bias, void *stream) {
    DirectArgs a = make_args(g, x, w, y, bias);
    const int64_t total = g.N * g.K * g.P * g.Q;
    if (total == 0) return CONV_OK;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (blocks > cap) blocks = cap;
    conv_direct_generic_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

// ---------------------------------------------------------------- dp4a
constexpr int kDp4aKB = 8;          // output channels per block
constexpr int kDp4aThreads = 128;   // pixels per block
constexpr int kDp4aMaxRed = 1024;   // largest C*R*S (rounded up to 4) it takes

bool dp4a_supported(const ConvGeom &g) { return ((g.C * g.R * g.S + 3) & ~3LL) <= kDp4aMaxRed; }

// Reduction element e = (c*R + r)*S + s, zero-padded to a multiple of 4.
__global__ void __launch_bounds__(kDp4aThreads) conv_direct_dp4a_kernel(const DirectArgs a, int red4) {
    __shared__ int32_t s_w[kDp4aKB][kDp4aMaxRed / 4];
    __shared__ long long s_off[kDp4aMaxRed];  // image offset of element e relative to (n, h0, w0)
    __shared__ int s_dh[kDp4aMaxRed];         // r*dil_h (or -1<<30 for padding elements)
    __shared__ int s_dw[kDp4aMaxRed];
    // (C*R*S <= kDp4aMaxRed: the reduction index and its tap fit 32 bits)
    const int red = (int)(a.C * a.R * a.S);
    const int S = (int)a.S, R = (int)a.R;
    const int64_t k0 = (int64_t)blockIdx.y * kDp4aKB;
    for (int e = threadIdx.x; e < red4 * 4; e += blockDim.x) {
        if (e < red) {
            const int s = e % S, r = (e / S) % R, c = e / (S * R);
            s_off[e] = c * a.xs1 + r * a.dil_h * a.xs2 + s * a.dil_w * a.xs3;
            s_dh[e] = (int)(r * a.dil_h);
            s_dw[e] = (int)(s * a.dil_w);
        } else {
            s_off[e] = 0;
            s_dh[e] = -(1 << 30);
            s_dw[e] = 0;
        }
    }
    for (int i = threadIdx.x; i < kDp4aKB * red4; i += blockDim.x) {
        const int kk = i / red4, u = i % red4;
        const int64_t k = k0 + kk;
        int8_t v[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int e = u * 4 + b;
            v[b] = 0;
            if (k < a.K && e < red) {
                const int s = e % S, r = (e / S) % R, c = e / (S * R);
                const int rf = a.mode ? R - 1 - r : r;
                const int sf = a.mode ? S - 1 - s : s;
                v[b] = __ldg(a.w + (k * a.ws0 + c * a.ws1 + rf * a.ws2 + sf * a.ws3));
            }
        }
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) word |= (uint32_t)(uint8_t)v[b] << (8 * b);
        s_w[kk][u] = (int32_t)word;
    }
    __syncthreads();
    const int64_t npix = a.N * a.P * a.Q;
    for (int64_t pix = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; pix < npix;
         pix += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = pix % a.Q;
        const int64_t t = pix / a.Q;
        const int64_t p = t % a.P;
        const int64_t n = t / a.P;
        const int64_t h0 = p * a.str_h - a.pad_h;
        const int64_t w0 = q * a.str_w - a.pad_w;
        // offset of the (possibly out-of-image) window origin; only in-image
        // elements are ever dereferenced
        const int64_t base = n * a.xs0 + h0 * a.xs2 + w0 * a.xs3;
        int32_t acc[kDp4aKB];
#pragma unroll
        for (int kk = 0; kk < kDp4aKB; ++kk) acc[kk] = 0;
        // four reduction words (16 image bytes) per round, all their loads
        // in flight together
        for (int u0 = 0; u0 < red4; u0 += 4) {
            int8_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int e = u0 * 4 + i;
                const int64_t h = h0 + s_dh[e < red4 * 4 ? e : 0];
                const int64_t w = w0 + s_dw[e < red4 * 4 ? e : 0];
                v[i] = 0;
                if (e < red4 * 4 && h >= 0 && h < a.H && w >= 0 && w < a.W) v[i] = __ldg(a.x + (base + s_off[e]));
            }
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
                if (u0 + uu >= red4) break;
                const uint32_t word = (uint32_t)(uint8_t)v[4 * uu] | ((uint32_t)(uint8_t)v[4 * uu + 1] << 8) |
                                      ((uint32_t)(uint8_t)v[4 * uu + 2] << 16) |
                                      ((uint32_t)(uint8_t)v[4 * uu + 3] << 24);
#pragma unroll
                for (int kk = 0; kk < kDp4aKB; ++kk) acc[kk] = __dp4a((int)word, s_w[kk][u0 + uu], acc[kk]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < kDp4aKB; ++kk) {
            const int64_t k = k0 + kk;
            if (k < a.K)
                store_out(a, n * a.ys0 + k * a.ys1 + p * a.ys2 + q * a.ys3, finish(acc[kk], a.bias, k, a.relu));
        }
    }
}

conv_status dp4a_launch(const ConvGeom &g, const int8_t *x, const int8_t *w, void *y,
                        const int32_t *bias, void *stream) {
    if (!dp4a_supported(g)) return CONV_ERR_ALIGNMENT;
    DirectArgs a = make_args(g, x, w, y, bias);
    const int64_t npix = g.N * g.P * g.Q;
    if (npix == 0 || g.K == 0) return CONV_OK;
    const int red4 = (int)((g.C * g.R * g.S + 3) / 4);
    const int64_t kblocks = (g.K + kDp4aKB - 1) / kDp4aKB;
    if (kblocks > 65535) return CONV_ERR_TOO_LARGE;
    int64_t pblocks = (npix + kDp4aThreads - 1) / kDp4aThreads;
    const int64_t cap = (int64_t)device_sm_count() * 32;
    if (pblocks > cap) pblocks = cap;
    dim3 grid((unsigned)pblocks, (unsigned)kblocks);
    conv_direct_dp4a_kernel<<<grid, kDp4aThreads, 0, (cudaStream_t)stream>>>(a, red4);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // namespace i8c
