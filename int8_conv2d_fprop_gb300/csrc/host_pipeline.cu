// host_pipeline.cu -- conv_fprop with the tensors in host memory.
//
// The batch is cut into a short lead chunk (a quarter of a chunk) and up
// to four chunks of whole images.  The filter and
// bias are copied once; then, on three library-owned streams, chunk c's image
// copy (host -> device) overlaps chunk c-1's convolution and chunk c-2's
// output copy (device -> host).  Device chunk buffers are double-buffered in
// the caller's device buffer.  Every image of a chunk must lie in one byte
// range of the host buffer, which holds when the batch dimension is the
// outermost one in memory (NCHW, NHWC and their padded variants); otherwise
// the whole batch is one chunk.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "internal.h"

namespace i8c {
namespace {

constexpr int kMaxChunks = 4;
constexpr int kMaxSlots = kMaxChunks + 1;  // plus the short lead chunk
constexpr int64_t kMinChunkBytes = 8 << 20;
constexpr int kMaxDevices = 64;

struct DeviceRes {
    std::mutex mu;  // one pipelined call per device at a time
    bool ready = false;
    cudaStream_t s_in = nullptr, s_cmp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_w = nullptr;
    cudaEvent_t ev_in[kMaxSlots] = {}, ev_cmp[kMaxSlots] = {}, ev_out[kMaxSlots] = {};
};
DeviceRes g_res[kMaxDevices];

conv_status init_res(DeviceRes &r) {
    if (r.ready) return CONV_OK;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    if (!ok(cudaStreamCreateWithFlags(&r.s_in, cudaStreamNonBlocking)) ||
        !ok(cudaStreamCreateWithFlags(&r.s_cmp, cudaStreamNonBlocking)) ||
        !ok(cudaStreamCreateWithFlags(&r.s_out, cudaStreamNonBlocking)) ||
        !ok(cudaEventCreateWithFlags(&r.ev_start, cudaEventDisableTiming)) ||
        !ok(cudaEventCreateWithFlags(&r.ev_w, cudaEventDisableTiming)))
        return CONV_ERR_CUDA;
    for (int i = 0; i < kMaxSlots; ++i) {
        if (!ok(cudaEventCreateWithFlags(&r.ev_in[i], cudaEventDisableTiming)) ||
            !ok(cudaEventCreateWithFlags(&r.ev_cmp[i], cudaEventDisableTiming)) ||
            !ok(cudaEventCreateWithFlags(&r.ev_out[i], cudaEventDisableTiming)))
            return CONV_ERR_CUDA;
    }
    r.ready = true;
    return CONV_OK;
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

// Extent, in elements, of the first `n` images of a descriptor.
int64_t extent_of_images(const conv_tensor_desc *d, int64_t n) {
    conv_tensor_desc t = *d;
    t.dims[0] = n;
    return desc_extent_elems(&t);
}

struct HostPlan {
    int chunks;
    int64_t per_chunk;       // images per chunk at most (the lead and the last chunk hold fewer)
    int64_t start[kMaxSlots + 1];  // chunk c covers images start[c] .. start[c+1]-1
    int64_t x_chunk_elems;   // device bytes of one image chunk
    int64_t y_chunk_elems;   // output elements of one output chunk
    int64_t y_esz;           // bytes per output element (4 for int32, 1 for int8)
    int64_t w_elems;
    size_t ws_bytes;         // conv workspace for one chunk
    size_t off_w, off_bias, off_ws, off_x[2], off_y[2], total;
};

conv_status host_plan(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                      const conv_fprop_params *p, HostPlan *hp) {
    const int64_t bias_elems = (p && (p->epilogue & CONV_EPILOGUE_BIAS)) && w ? w->dims[0] : 0;
    conv_status st = conv_fprop_validate(x, w, y, p, bias_elems);
    if (st) return st;
    const int64_t N = x->dims[0];
    hp->y_esz = (p->epilogue & CONV_EPILOGUE_INT8_OUT) ? 1 : 4;
    // whole images in disjoint, ordered byte ranges?
    const bool batch_outer = N <= 1 || (x->strides[0] >= extent_of_images(x, 1) &&
                                        y->strides[0] >= extent_of_images(y, 1));
    // chunks only pay off when each moves a good amount of data: at least
    // kMinChunkBytes of output per chunk
    int64_t max_chunks = N < kMaxChunks ? N : kMaxChunks;
    const int64_t y_bytes = desc_extent_elems(y) * hp->y_esz;
    while (max_chunks > 1 && y_bytes / max_chunks < kMinChunkBytes) --max_chunks;
    hp->chunks = (!batch_outer || N < 2) ? 1 : (int)max_chunks;
    hp->per_chunk = N == 0 ? 0 : (N + hp->chunks - 1) / hp->chunks;
    // rounding the chunk size up can leave fewer non-empty chunks (N = 5 in
    // chunks of 2 needs 3, not 4)
    if (N > 0) hp->chunks = (int)((N + hp->per_chunk - 1) / hp->per_chunk);
    // a short lead chunk (a quarter of a chunk) first: the output's copy to
    // the host, the longest stage (the link moves about 190 GB/s to the host
    // whatever does the copy), starts after it instead of after a full chunk
    hp->start[0] = 0;
    if (hp->chunks > 1 && hp->per_chunk >= 2) {
        int c = 0;
        hp->start[++c] = hp->per_chunk / 4 > 0 ? hp->per_chunk / 4 : 1;
        while (hp->start[c] < N) {
            const int64_t nxt = hp->start[c] + hp->per_chunk;
            hp->start[c + 1] = nxt < N ? nxt : N;
            ++c;
        }
        hp->chunks = c;
    } else {
        for (int c = 0; c < hp->chunks; ++c) {
            const int64_t nxt = (int64_t)(c + 1) * hp->per_chunk;
            hp->start[c + 1] = nxt < N ? nxt : N;
        }
    }
    hp->x_chunk_elems = hp->chunks == 1 ? desc_extent_elems(x) : extent_of_images(x, hp->per_chunk);
    hp->y_chunk_elems = hp->chunks == 1 ? desc_extent_elems(y) : extent_of_images(y, hp->per_chunk);
    hp->w_elems = desc_extent_elems(w);
    conv_tensor_desc xc = *x, yc = *y;
    xc.dims[0] = yc.dims[0] = hp->per_chunk;
    xc.capacity_bytes = (uint64_t)hp->x_chunk_elems;
    yc.capacity_bytes = (uint64_t)(hp->y_chunk_elems * hp->y_esz);
    hp->ws_bytes = 0;
    if (hp->per_chunk > 0 && (st = conv_fprop_workspace_size(&xc, w, &yc, p, &hp->ws_bytes))) return st;
    // the lead and the last chunk may hold fewer images, and with fewer
    // tiles their plans may cut tiles along the reduction where the full
    // chunks' plan does not: the workspace serves every chunk size
    for (int c = 0; hp->chunks > 1 && c < hp->chunks; ++c) {
        const int64_t nb = hp->start[c + 1] - hp->start[c];
        if (nb == hp->per_chunk) continue;
        conv_tensor_desc xl = *x, yl = *y;
        xl.dims[0] = yl.dims[0] = nb;
        xl.capacity_bytes = (uint64_t)extent_of_images(x, nb);
        yl.capacity_bytes = (uint64_t)(extent_of_images(y, nb) * hp->y_esz);
        size_t wl = 0;
        if ((st = conv_fprop_workspace_size(&xl, w, &yl, p, &wl))) return st;
        if (wl > hp->ws_bytes) hp->ws_bytes = wl;
    }
    size_t off = 0;
    hp->off_w = off;
    off = align256(off + (size_t)hp->w_elems);
    hp->off_bias = off;
    off = align256(off + (size_t)bias_elems * 4);
    hp->off_ws = off;
    off = align256(off + hp->ws_bytes);
    for (int b = 0; b < 2; ++b) {
        hp->off_x[b] = off;
        off = align256(off + (size_t)hp->x_chunk_elems);
    }
    for (int b = 0; b < 2; ++b) {
        hp->off_y[b] = off;
        off = align256(off + (size_t)(hp->y_chunk_elems * hp->y_esz));
    }
    hp->total = off;
    return CONV_OK;
}

}  // namespace
}  // namespace i8c

using namespace i8c;

extern "C" {

conv_status conv_fprop_host_buffer_size(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                        const conv_tensor_desc *y, const conv_fprop_params *p, size_t *bytes) {
    if (!bytes) return CONV_ERR_NULL_PTR;
    HostPlan hp;
    conv_status st = host_plan(x, w, y, p, &hp);
    if (st) return st;
    *bytes = hp.total;
    return CONV_OK;
}

conv_status conv_fprop_host(const conv_tensor_desc *x, const int8_t *x_host, const conv_tensor_desc *w,
                            const int8_t *w_host, const conv_tensor_desc *y, void *y_host,
                            const int32_t *bias_host, const conv_fprop_params *p, void *device_buffer,
                            size_t device_buffer_bytes, void *stream) {
    HostPlan hp;
    conv_status st = host_plan(x, w, y, p, &hp);
    if (st) return st;
    if (x->dims[0] == 0 || w->dims[0] == 0) return CONV_OK;
    const bool bias = (p->epilogue & CONV_EPILOGUE_BIAS) != 0;
    if (!x_host || !w_host || !y_host || !device_buffer || (bias && !bias_host)) return CONV_ERR_NULL_PTR;
    if (device_buffer_bytes < hp.total || ((uintptr_t)device_buffer % 256) != 0) return CONV_ERR_WORKSPACE;
    if ((st = check_device())) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CONV_ERR_CUDA;
    DeviceRes &r = g_res[dev];
    std::lock_guard<std::mutex> lock(r.mu);
    if ((st = init_res(r))) return st;

    uint8_t *buf = static_cast<uint8_t *>(device_buffer);
    int8_t *w_dev = reinterpret_cast<int8_t *>(buf + hp.off_w);
    int32_t *b_dev = bias ? reinterpret_cast<int32_t *>(buf + hp.off_bias) : nullptr;
    void *ws = hp.ws_bytes ? buf + hp.off_ws : nullptr;
    cudaStream_t caller = (cudaStream_t)stream;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };

    if (!ok(cudaEventRecord(r.ev_start, caller)) || !ok(cudaStreamWaitEvent(r.s_in, r.ev_start, 0)) ||
        !ok(cudaStreamWaitEvent(r.s_cmp, r.ev_start, 0)) || !ok(cudaStreamWaitEvent(r.s_out, r.ev_start, 0)))
        return CONV_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(w_dev, w_host, (size_t)hp.w_elems, cudaMemcpyHostToDevice, r.s_in)))
        return CONV_ERR_CUDA;
    if (bias && !ok(cudaMemcpyAsync(b_dev, bias_host, (size_t)w->dims[0] * 4, cudaMemcpyHostToDevice, r.s_in)))
        return CONV_ERR_CUDA;
    if (!ok(cudaEventRecord(r.ev_w, r.s_in)) || !ok(cudaStreamWaitEvent(r.s_cmp, r.ev_w, 0))) return CONV_ERR_CUDA;

    for (int c = 0; c < hp.chunks; ++c) {
        const int bsel = c & 1;
        const int64_t n0 = hp.start[c];
        const int64_t nb = hp.start[c + 1] - n0;
        if (nb <= 0) return CONV_ERR_BAD_PARAM;  // cannot happen: the starts increase
        conv_tensor_desc xc = *x, yc = *y;
        xc.dims[0] = yc.dims[0] = nb;
        const int64_t x_elems = hp.chunks == 1 ? desc_extent_elems(x) : extent_of_images(x, nb);
        const int64_t y_elems = hp.chunks == 1 ? desc_extent_elems(y) : extent_of_images(y, nb);
        xc.capacity_bytes = (uint64_t)x_elems;
        yc.capacity_bytes = (uint64_t)(y_elems * hp.y_esz);
        int8_t *x_dev = reinterpret_cast<int8_t *>(buf + hp.off_x[bsel]);
        void *y_dev = buf + hp.off_y[bsel];
        // image chunk in; its buffer was last read by the convolution of chunk c-2
        if (c >= 2 && !ok(cudaStreamWaitEvent(r.s_in, r.ev_cmp[c - 2], 0))) return CONV_ERR_CUDA;
        if (!ok(cudaMemcpyAsync(x_dev, x_host + n0 * x->strides[0], (size_t)x_elems, cudaMemcpyHostToDevice,
                                r.s_in)) ||
            !ok(cudaEventRecord(r.ev_in[c], r.s_in)))
            return CONV_ERR_CUDA;
        // convolution; its output buffer was last read by the copy-out of chunk c-2
        if (!ok(cudaStreamWaitEvent(r.s_cmp, r.ev_in[c], 0))) return CONV_ERR_CUDA;
        if (c >= 2 && !ok(cudaStreamWaitEvent(r.s_cmp, r.ev_out[c - 2], 0))) return CONV_ERR_CUDA;
        if (c == 0 && (st = conv_fprop_pack_filter(&xc, w, w_dev, &yc, p, ws, hp.ws_bytes, r.s_cmp))) return st;
        if ((st = conv_fprop_prepacked(&xc, x_dev, w, w_dev, &yc, y_dev, b_dev, p, ws, hp.ws_bytes, r.s_cmp)))
            return st;
        if (!ok(cudaEventRecord(r.ev_cmp[c], r.s_cmp))) return CONV_ERR_CUDA;
        // output chunk out
        if (!ok(cudaStreamWaitEvent(r.s_out, r.ev_cmp[c], 0)) ||
            !ok(cudaMemcpyAsync(static_cast<uint8_t *>(y_host) + n0 * y->strides[0] * hp.y_esz, y_dev,
                                (size_t)(y_elems * hp.y_esz), cudaMemcpyDeviceToHost, r.s_out)) ||
            !ok(cudaEventRecord(r.ev_out[c], r.s_out)))
            return CONV_ERR_CUDA;
    }
    // the caller's stream resumes once the last output chunk is home (which
    // orders after every earlier copy and convolution)
    if (!ok(cudaStreamWaitEvent(caller, r.ev_out[hp.chunks - 1], 0))) return CONV_ERR_CUDA;
    return CONV_OK;
}

}  // extern "C"
