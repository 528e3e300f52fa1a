// api.cu -- the conv_fprop entry points: validation, planning, dispatch to
// the kernels, the device status word and the timeout self-test.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

namespace i8c {

// One status word per device (every device that loads the module holds its
// own copy).  Kernels write CONV_ERR_DEVICE_TIMEOUT here when a wait expires.
__device__ int g_conv_device_status = 0;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_ok[kMaxDevices];    // 0 unknown, 1 sm_103, 2 other
std::atomic<int> g_dev_sms[kMaxDevices];
std::atomic<int *> g_dev_status[kMaxDevices];
}  // namespace

int *device_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int *ptr = g_dev_status[dev].load();
    if (!ptr) {
        // host code must not take the address of a __device__ variable
        // directly; ask the runtime for this device's copy
        if (cudaGetSymbolAddress((void **)&ptr, g_conv_device_status) != cudaSuccess) return nullptr;
        g_dev_status[dev].store(ptr);
    }
    return ptr;
}

conv_status check_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CONV_ERR_UNSUPPORTED_DEVICE;
    int st = g_dev_ok[dev].load();
    if (st == 0) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return CONV_ERR_CUDA;
        st = (prop.major == 10 && prop.minor == 3) ? 1 : 2;
        g_dev_sms[dev].store(prop.multiProcessorCount);
        g_dev_ok[dev].store(st);
    }
    return st == 1 ? CONV_OK : CONV_ERR_UNSUPPORTED_DEVICE;
}

int device_sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    int n = (dev >= 0 && dev < kMaxDevices) ? g_dev_sms[dev].load() : 0;
    if (n <= 0) {
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

uint64_t wait_limit_ns() {
    static const uint64_t v = [] {
        const char *e = std::getenv("INT8CONV_WAIT_LIMIT_MS");
        long ms = e ? std::atol(e) : 1000;
        if (ms < 1) ms = 1;
        if (ms > 60000) ms = 60000;
        return (uint64_t)ms * 1000000ull;
    }();
    return v;
}

static void put_desc(PlanKey &k, const conv_tensor_desc *d) {
    k.v[k.n++] = d->dtype;
    k.v[k.n++] = d->rank;
    for (int i = 0; i < 4; ++i) k.v[k.n++] = d->dims[i];
    for (int i = 0; i < 4; ++i) k.v[k.n++] = d->strides[i];
    k.v[k.n++] = (int64_t)d->capacity_bytes;
}

PlanKey make_plan_key(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                      const conv_fprop_params *p, const void *x_dev, int dev) {
    PlanKey k;
    std::memset(&k, 0, sizeof(k));
    put_desc(k, x);
    put_desc(k, w);
    put_desc(k, y);
    for (int i = 0; i < 2; ++i) {
        k.v[k.n++] = p->pre_padding[i];
        k.v[k.n++] = p->post_padding[i];
        k.v[k.n++] = p->stride[i];
        k.v[k.n++] = p->dilation[i];
    }
    k.v[k.n++] = p->mode;
    k.v[k.n++] = p->compute_dtype;
    k.v[k.n++] = p->epilogue;
    k.v[k.n++] = p->algo;
    k.v[k.n++] = p->out_shift;
    k.v[k.n++] = dev;
    k.v[k.n++] = (x_dev == nullptr || ((uintptr_t)x_dev % 16) == 0) ? 1 : 0;
    return k;
}


namespace {

int choose_algo(const ConvGeom &g, int requested) {
    if (requested != CONV_ALGO_AUTO) return requested;
    if (g.C >= 16 && igemm_supported(g)) return CONV_ALGO_IMPLICIT_GEMM;
    if (dp4a_supported(g)) return CONV_ALGO_DIRECT_DP4A;
    if (igemm_supported(g)) return CONV_ALGO_IMPLICIT_GEMM;
    return CONV_ALGO_DIRECT_GENERIC;
}

// Plan cache: the validated geometry, algorithm and tensor-core plan of a
// call, keyed by its descriptors, parameters, device and whether the image
// pointer is 16-byte aligned (the only thing the plan reads of a pointer).
// Repeated calls with the same shapes skip validation and planning.  Least
// recently used entries give way; conv_shutdown empties it.
constexpr int kPlanCacheSize = 64;
struct PlanCacheEntry {
    PlanKey key;
    ConvGeom g;
    int algo;
    IgemmPlan pl;
    uint64_t used;
    bool valid;
};
std::mutex g_plan_mu;
PlanCacheEntry g_plan_cache[kPlanCacheSize];
uint64_t g_plan_clock = 0;
std::atomic<uint64_t> g_plan_hits{0}, g_plan_misses{0};

conv_status plan_call_uncached(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                               const conv_fprop_params *p, const void *x_dev, ConvGeom *g, int *algo,
                               IgemmPlan *pl);

conv_status plan_call(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                      const conv_fprop_params *p, const void *x_dev, ConvGeom *g, int *algo, IgemmPlan *pl) {
    if (!x || !w || !y || !p) return CONV_ERR_NULL_PTR;
    int dev = 0;
    cudaGetDevice(&dev);  // (no device: plans are keyed on ordinal 0)
    const PlanKey key = make_plan_key(x, w, y, p, x_dev, dev);
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        for (auto &e : g_plan_cache)
            if (e.valid && e.key.n == key.n && std::memcmp(e.key.v, key.v, sizeof(int64_t) * key.n) == 0) {
                e.used = ++g_plan_clock;
                *g = e.g;
                *algo = e.algo;
                *pl = e.pl;
                g_plan_hits.fetch_add(1);
                return CONV_OK;
            }
    }
    g_plan_misses.fetch_add(1);
    conv_status st = plan_call_uncached(x, w, y, p, x_dev, g, algo, pl);
    if (st) return st;  // only valid plans are kept
    std::lock_guard<std::mutex> lock(g_plan_mu);
    PlanCacheEntry *victim = &g_plan_cache[0];
    for (auto &e : g_plan_cache) {
        if (!e.valid) {
            victim = &e;
            break;
        }
        if (e.used < victim->used) victim = &e;
    }
    victim->key = key;
    victim->g = *g;
    victim->algo = *algo;
    victim->pl = *pl;
    victim->used = ++g_plan_clock;
    victim->valid = true;
    return CONV_OK;
}

conv_status plan_call_uncached(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                               const conv_fprop_params *p, const void *x_dev, ConvGeom *g, int *algo,
                               IgemmPlan *pl) {
    const int64_t bias_elems = (p && (p->epilogue & CONV_EPILOGUE_BIAS)) ? (w ? w->dims[0] : 0) : 0;
    conv_status st = conv_fprop_validate(x, w, y, p, bias_elems);
    if (st) return st;
    make_geom(x, w, y, p, g);
    const bool global_loads = p->algo == CONV_ALGO_IMPLICIT_GEMM_GLOBAL_LOADS;
    *algo = choose_algo(*g, global_loads ? CONV_ALGO_IMPLICIT_GEMM : p->algo);
    if (*algo == CONV_ALGO_IMPLICIT_GEMM && !igemm_supported(*g)) return CONV_ERR_ALIGNMENT;
    if (*algo == CONV_ALGO_DIRECT_DP4A && !dp4a_supported(*g)) return CONV_ERR_ALIGNMENT;
    if (*algo == CONV_ALGO_IMPLICIT_GEMM) {
        igemm_plan(*g, x_dev, pl, global_loads);
    }
    return CONV_OK;
}

__global__ void selftest_wait_kernel(uint64_t limit_ns, int *status) {
    __shared__ uint64_t bar;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nobody arrives on this barrier: the wait must run out, record the
        // timeout and return
        const uint64_t t0 = ptx::global_timer_ns();
        while (!ptx::mbar_try_wait(b, 0)) {
            if (ptx::global_timer_ns() - t0 > limit_ns) {
                atomicExch(status, (int)CONV_ERR_DEVICE_TIMEOUT);
                break;
            }
        }
        // complete the phase so the barrier is left in a clean state
        ptx::mbar_arrive(b);
    }
    __syncthreads();
}

}  // namespace

conv_status conv_fprop_workspace_size_for(const conv_tensor_desc *x, const void *x_dev, const conv_tensor_desc *w,
                                          const conv_tensor_desc *y, const conv_fprop_params *p, size_t *bytes) {
    if (!bytes) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, x_dev, &g, &algo, &pl);
    if (st) return st;
    *bytes = (algo == CONV_ALGO_IMPLICIT_GEMM && g.N > 0 && g.K > 0) ? pl.workspace_bytes : 0;
    return CONV_OK;
}

}  // namespace i8c

using namespace i8c;

extern "C" {

conv_status conv_fprop_plan(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                            const conv_fprop_params *p, int32_t *algo_out) {
    if (!algo_out) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, nullptr, &g, &algo, &pl);
    if (st) return st;
    *algo_out = (algo == CONV_ALGO_IMPLICIT_GEMM && pl.register_loads) ? CONV_ALGO_IMPLICIT_GEMM_GLOBAL_LOADS : algo;
    return CONV_OK;
}

conv_status conv_fprop_workspace_size(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                      const conv_tensor_desc *y, const conv_fprop_params *p, size_t *bytes) {
    if (!bytes) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, nullptr, &g, &algo, &pl);
    if (st) return st;
    // the image pointer is assumed 16-byte aligned here (see the header)
    *bytes = algo == CONV_ALGO_IMPLICIT_GEMM ? pl.workspace_bytes : 0;
    return CONV_OK;
}

conv_status conv_fprop_kernel_count(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                    const conv_tensor_desc *y, const conv_fprop_params *p, int32_t *count) {
    if (!count) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, nullptr, &g, &algo, &pl);
    if (st) return st;
    if (g.N == 0 || g.K == 0 || g.P == 0 || g.Q == 0) {
        *count = 0;
    } else if (algo != CONV_ALGO_IMPLICIT_GEMM) {
        *count = 1;
    } else {
        *count = (igemm_filter_in_kernel(g, pl, nullptr) ? 1 : 2) + (pl.pack_x ? 1 : 0) + (pl.splits > 1 ? 1 : 0);
    }
    return CONV_OK;
}

conv_status conv_fprop_tile_shape(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                  const conv_tensor_desc *y, const conv_fprop_params *p, int64_t shape[4]) {
    if (!shape) return CONV_ERR_NULL_PTR;
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, nullptr, &g, &algo, &pl);
    if (st) return st;
    for (int i = 0; i < 4; ++i) shape[i] = 0;
    if (g.N == 0 || g.K == 0 || g.P == 0 || g.Q == 0 || algo != CONV_ALGO_IMPLICIT_GEMM) return CONV_OK;
    shape[0] = kIgemmMTile;
    shape[1] = pl.n_tile;
    shape[2] = pl.m_tiles * pl.n_tiles;
    shape[3] = pl.num_units;
    return CONV_OK;
}

namespace {

// Validation, planning and pointer checks shared by the three entry points
// that launch work.  *nothing_to_do is set for an empty output.
conv_status prepare_call(const conv_tensor_desc *x, const int8_t *x_dev, const conv_tensor_desc *w,
                         const int8_t *w_dev, const conv_tensor_desc *y, void *y_dev, const int32_t *bias_dev,
                         const conv_fprop_params *p, void *workspace, size_t workspace_bytes, ConvGeom *g,
                         int *algo, IgemmPlan *pl, bool *nothing_to_do) {
    conv_status st = plan_call(x, w, y, p, x_dev, g, algo, pl);
    if (st) return st;
    *nothing_to_do = (g->N == 0 || g->K == 0);
    if (*nothing_to_do) return CONV_OK;
    if (!x_dev || !w_dev || !y_dev) return CONV_ERR_NULL_PTR;
    if (g->bias && !bias_dev) return CONV_ERR_NULL_PTR;
    const uint64_t ybytes = (uint64_t)desc_extent_elems(y) * (g->out_int8 ? 1u : 4u);
    if (overlaps(y_dev, ybytes, x_dev, (uint64_t)desc_extent_elems(x)) ||
        overlaps(y_dev, ybytes, w_dev, (uint64_t)desc_extent_elems(w)) ||
        overlaps(y_dev, ybytes, workspace, workspace_bytes) ||
        (g->bias && overlaps(y_dev, ybytes, bias_dev, (uint64_t)g->K * 4)))
        return CONV_ERR_OVERLAP;
    if (*algo == CONV_ALGO_IMPLICIT_GEMM) {
        if (!workspace || workspace_bytes < pl->workspace_bytes || ((uintptr_t)workspace % 256) != 0)
            return CONV_ERR_WORKSPACE;
        if (overlaps(workspace, pl->workspace_bytes, x_dev, (uint64_t)desc_extent_elems(x)) ||
            overlaps(workspace, pl->workspace_bytes, w_dev, (uint64_t)desc_extent_elems(w)))
            return CONV_ERR_OVERLAP;
    }
    return check_device();
}

conv_status run_main(const ConvGeom &g, int algo, const IgemmPlan &pl, const int8_t *x_dev, const int8_t *w_dev,
                     void *y_dev, const int32_t *bias_dev, void *workspace, void *stream, bool repack) {
    switch (algo) {
        case CONV_ALGO_IMPLICIT_GEMM:
            return igemm_main_launch(g, pl, x_dev, w_dev, y_dev, bias_dev, workspace, stream, repack);
        case CONV_ALGO_DIRECT_DP4A:
            return dp4a_launch(g, x_dev, w_dev, y_dev, bias_dev, stream);
        default:
            return generic_launch(g, x_dev, w_dev, y_dev, bias_dev, stream);
    }
}

}  // namespace

conv_status conv_fprop(const conv_tensor_desc *x, const int8_t *x_dev, const conv_tensor_desc *w,
                       const int8_t *w_dev, const conv_tensor_desc *y, void *y_dev, const int32_t *bias_dev,
                       const conv_fprop_params *p, void *workspace, size_t workspace_bytes, void *stream) {
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    bool none = false;
    conv_status st = prepare_call(x, x_dev, w, w_dev, y, y_dev, bias_dev, p, workspace, workspace_bytes, &g,
                                  &algo, &pl, &none);
    if (st || none) return st;
    // (the filter is repacked first unless the kernel converts it itself)
    return run_main(g, algo, pl, x_dev, w_dev, y_dev, bias_dev, workspace, stream, true);
}

conv_status conv_fprop_pack_filter(const conv_tensor_desc *x, const conv_tensor_desc *w, const int8_t *w_dev,
                                   const conv_tensor_desc *y, const conv_fprop_params *p, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    conv_status st = plan_call(x, w, y, p, nullptr, &g, &algo, &pl);
    if (st) return st;
    if (algo != CONV_ALGO_IMPLICIT_GEMM || g.N == 0 || g.K == 0) return CONV_OK;
    if (!w_dev) return CONV_ERR_NULL_PTR;
    if (!workspace || workspace_bytes < pl.wpack_bytes || ((uintptr_t)workspace % 256) != 0)
        return CONV_ERR_WORKSPACE;
    if (overlaps(workspace, pl.wpack_bytes, w_dev, (uint64_t)desc_extent_elems(w))) return CONV_ERR_OVERLAP;
    if ((st = check_device())) return st;
    return igemm_pack_filter_launch(g, pl, w_dev, workspace, stream);
}

conv_status conv_fprop_prepacked(const conv_tensor_desc *x, const int8_t *x_dev, const conv_tensor_desc *w,
                                 const int8_t *w_dev, const conv_tensor_desc *y, void *y_dev,
                                 const int32_t *bias_dev, const conv_fprop_params *p, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    ConvGeom g;
    IgemmPlan pl;
    int algo = 0;
    bool none = false;
    conv_status st = prepare_call(x, x_dev, w, w_dev, y, y_dev, bias_dev, p, workspace, workspace_bytes, &g,
                                  &algo, &pl, &none);
    if (st || none) return st;
    return run_main(g, algo, pl, x_dev, w_dev, y_dev, bias_dev, workspace, stream, false);
}

conv_status conv_device_status(void *stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return CONV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_conv_device_status, sizeof(int)) != cudaSuccess) return CONV_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_conv_device_status, &zero, sizeof(int)) != cudaSuccess) return CONV_ERR_CUDA;
    }
    return (conv_status)v;
}

void conv_shutdown(void) {
    {
        std::lock_guard<std::mutex> lock(g_plan_mu);
        for (auto &e : g_plan_cache) e.valid = false;
    }
    igemm_cache_clear();
    dgrad_cache_clear();
}

conv_status conv_plan_cache_stats(uint64_t *plan_hits, uint64_t *plan_misses, uint64_t *launch_hits,
                                  uint64_t *launch_misses) {
    if (!plan_hits || !plan_misses || !launch_hits || !launch_misses) return CONV_ERR_NULL_PTR;
    *plan_hits = g_plan_hits.load();
    *plan_misses = g_plan_misses.load();
    igemm_cache_stats(launch_hits, launch_misses);
    return CONV_OK;
}

conv_status conv_selftest_wait_timeout(uint32_t limit_us, void *stream) {
    conv_status st = check_device();
    if (st) return st;
    if (limit_us < 1 || limit_us > 2000000) return CONV_ERR_BAD_PARAM;
    int *status = device_status_word();
    if (!status) return CONV_ERR_CUDA;
    selftest_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_us * 1000ull, status);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // extern "C"
