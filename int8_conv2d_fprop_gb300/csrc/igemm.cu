// igemm.cu -- implicit-GEMM INT8 convolution on the sm_103a tensor cores.
//
// GEMM view of conv_fprop (cuDNN "Convolutions", section "Convolution
// Fprop"): rows m = output pixels (n, p, q), columns = output channels k,
// reduction = (r, s, c) taps x channels.  A[m, (r,s,c)] is the image pixel
// read at h = p*stride_h - pre_h + r*dil_h, w = q*stride_w - pre_w + s*dil_w
// (zero outside the image); B[k, (r,s,c)] is the filter, flipped in r and s
// for CONVOLUTION mode.
//
// sm_103a has no integer kind for tcgen05.mma, so the product is formed on the
// f16 path, exactly: every int8 value is an exact f16, every product of two
// (|x*w| <= 2^14) is exact, and an f32 sum of integers stays exact while its
// magnitude stays within 2^24.  The reduction is therefore cut into groups of
// at most 1024 terms (1024 * 2^14 = 2^24), each accumulated in its own tensor
// memory slot, converted to int32 by the epilogue warps and summed in int32
// registers.  The result is bit-identical to integer arithmetic.
//
// Persistent, warp-specialised CTA (one per SM), 512 threads, tile 128 pixels
// x NT output channels (NT = 128 or 256):
//   warpgroup 0  producers: each thread owns one pixel row of the A tile; it
//                gathers 64 channels of one tap with 16-byte loads (the im2col
//                address formed on the fly from stride, padding and
//                dilation), two items ahead of the one it stores, converts
//                int8 -> f16 in registers and writes the row into the
//                128-byte-swizzled shared-memory stage.  Thread 0 also brings
//                the matching pre-swizzled f16 filter block with one bulk
//                async copy.
//   warpgroup 1  warp 4 allocates tensor memory; its lane 0 issues
//                tcgen05.mma (M=128, N=NT, K=16 per instruction) into one of
//                two accumulator slots.  Warps 5-7 have no role.
//   warpgroups 2-3  epilogue, two warps per tensor-memory lane quadrant, each
//                owning NT/2 columns: tcgen05.ld each finished slot,
//                f32 -> int32, sum the groups, add bias, ReLU, store int32.
// Registers are moved from warpgroups 0-1 to the epilogue with setmaxnreg.
// Every wait is bounded in time; on expiry the CTA records
// CONV_ERR_DEVICE_TIMEOUT, stops, lets issued copies and MMAs finish and frees
// its tensor memory.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "tc_ptx.cuh"

namespace i8c {

namespace {

constexpr int MT = kIgemmMTile;  // 128
constexpr int KS = kIgemmKStep;  // 64 channels = 128 bytes of f16 per row
constexpr int NSLOT = 2;
constexpr int MAX_GROUP_STEPS = 1024 / KS;  // 16 k-steps: at most 1024 products per f32 sum
constexpr int A_BYTES = MT * KS * 2;       // 16 KB
constexpr int THREADS = 512;
constexpr int MMA_WARP = 4;
constexpr int FIRST_EPI_WARP = 8;
constexpr int NUM_EPI_THREADS = 256;
constexpr int PRODUCER_REGS = 80;
constexpr int EPILOGUE_REGS = 176;
static_assert(2 * 128 * PRODUCER_REGS + 2 * 128 * EPILOGUE_REGS <= 65536, "register split exceeds the launch");
constexpr int PREFETCH = 2;  // items in flight ahead of the one being stored

template <int NT>
struct TileCfg {
    static constexpr int B_BYTES = NT * KS * 2;
    static constexpr int STAGES = NT == 256 ? 4 : 6;
    static constexpr int TMEM_COLS = NSLOT * NT;
    static constexpr int SMEM_BYTES = 1024 /*align slack*/ + STAGES * (A_BYTES + B_BYTES) + 256 /*barriers*/;
    static_assert(TMEM_COLS <= 512, "tensor memory has 512 columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};

struct IgemmArgs {
    const int8_t *x;     // channels-last image
    const uint8_t *wp;   // repacked f16 filter blocks
    int32_t *y;
    const int32_t *bias;
    int64_t xs_n, xs_h, xs_w;  // element (= byte) strides of the channels-last image
    int64_t ys_n, ys_k, ys_p, ys_q;
    int32_t H, W, P, Q, K, S;
    int32_t c16;         // channel bytes per pixel that may be loaded (multiple of 16)
    int32_t c_steps, k_steps, groups;
    int32_t pad_h, pad_w, str_h, str_w, dil_h, dil_w;
    int32_t m_total, n_tiles, num_tiles;
    int32_t relu, y_vec;
    uint64_t wait_limit_ns;
    int *status;         // device status word
};

template <int STAGES>
struct SharedCtl {
    uint64_t a_full[STAGES];
    uint64_t b_full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[NSLOT];
    uint64_t acc_empty[NSLOT];
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(SharedCtl<6>) <= 256, "control block too large");

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// the time limit passed (then the CTA is marked aborting and the device status
// word records the timeout).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int32_t *abort_flag,
                                           uint64_t limit_ns, int *status) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicExch(status, (int)CONV_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag: used while shutting down to let
// work already issued (bulk copies, MMAs) finish before shared or tensor
// memory is released.
__device__ __forceinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns, int *status) {
    const uint64_t t0 = ptx::global_timer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::global_timer_ns() - t0 > limit_ns) {
            atomicExch(status, (int)CONV_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
    return true;
}

// 16 int8 -> 16 f16 (two 16-byte chunks).  x ^ 0x80 turns each signed byte
// into u = x + 128; placing u under the f16 exponent of 1024 gives 1024 + u,
// and subtracting 1152 leaves x exactly.
__device__ __forceinline__ uint32_t cvt_pair(uint32_t word_xor, uint32_t sel) {
    const uint32_t h2 = __byte_perm(word_xor, 0x64646464u, sel);
    __half2 v = *reinterpret_cast<const __half2 *>(&h2);
    v = __hsub2(v, __half2half2(__ushort_as_half((unsigned short)0x6480)));  // 1152.0
    return *reinterpret_cast<const uint32_t *>(&v);
}

__device__ __forceinline__ void cvt16(const uint4 in, uint4 &lo, uint4 &hi) {
    const uint32_t a = in.x ^ 0x80808080u, b = in.y ^ 0x80808080u;
    const uint32_t c = in.z ^ 0x80808080u, d = in.w ^ 0x80808080u;
    lo.x = cvt_pair(a, 0x4140); lo.y = cvt_pair(a, 0x4342);
    lo.z = cvt_pair(b, 0x4140); lo.w = cvt_pair(b, 0x4342);
    hi.x = cvt_pair(c, 0x4140); hi.y = cvt_pair(c, 0x4342);
    hi.z = cvt_pair(d, 0x4140); hi.w = cvt_pair(d, 0x4342);
}

// Where one producer thread is in its (tile, k-step) sequence.
struct LoadCursor {
    int tile;       // tile index, >= num_tiles when done
    int j, cb, r, s;
    int64_t xoff;   // n * xs_n
    int h0, w0;
    bool valid;     // this thread's pixel row exists
};

__device__ __forceinline__ void cursor_set_tile(LoadCursor &c, const IgemmArgs &a, int tile, int row) {
    c.tile = tile;
    c.j = c.cb = c.r = c.s = 0;
    const int mt = tile / a.n_tiles;
    const int m = mt * MT + row;
    c.valid = tile < a.num_tiles && m < a.m_total;
    const int mm = c.valid ? m : 0;
    const int pq = a.P * a.Q;
    const int n = mm / pq;
    const int rem = mm - n * pq;
    const int p = rem / a.Q;
    const int q = rem - p * a.Q;
    c.xoff = (int64_t)n * a.xs_n;
    c.h0 = p * a.str_h - a.pad_h;
    c.w0 = q * a.str_w - a.pad_w;
}

__device__ __forceinline__ void cursor_load(const LoadCursor &c, const IgemmArgs &a, uint4 (&v)[4]) {
    const int h = c.h0 + c.r * a.dil_h;
    const int w = c.w0 + c.s * a.dil_w;
    const bool ok = c.valid && (unsigned)h < (unsigned)a.H && (unsigned)w < (unsigned)a.W;
    const int cbase = c.cb * KS;
    const int8_t *src = a.x + (c.xoff + (int64_t)h * a.xs_h + (int64_t)w * a.xs_w + cbase);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (ok && cbase + 16 * i < a.c16)
            v[i] = ptx::ld_nc_v4(src + 16 * i);
        else
            v[i] = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ void cursor_advance(LoadCursor &c, const IgemmArgs &a, int row) {
    if (++c.j == a.k_steps) {
        cursor_set_tile(c, a, c.tile + gridDim.x, row);
        return;
    }
    if (++c.cb == a.c_steps) {
        c.cb = 0;
        if (++c.s == a.S) {
            c.s = 0;
            ++c.r;
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(THREADS, 1) igemm_conv_kernel(const __grid_constant__ IgemmArgs a) {
    using Cfg = TileCfg<NT>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int B_BYTES = Cfg::B_BYTES;
    constexpr int HALF = NT / 2;  // columns per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const uint32_t a_smem = base;
    const uint32_t b_smem = base + STAGES * A_BYTES;
    SharedCtl<STAGES> *ctl = reinterpret_cast<SharedCtl<STAGES> *>(base_ptr + STAGES * (A_BYTES + B_BYTES));
    volatile int32_t *abort_flag = &ctl->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            ptx::mbar_init(ptx::smem_addr(&ctl->a_full[i]), 128);
            ptx::mbar_init(ptx::smem_addr(&ctl->b_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->empty[i]), 1);
        }
        for (int i = 0; i < NSLOT; ++i) {
            ptx::mbar_init(ptx::smem_addr(&ctl->acc_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->acc_empty[i]), NUM_EPI_THREADS);
        }
        ptx::mbar_init(ptx::smem_addr(&ctl->mma_done), 1);
        ctl->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        ptx::tmem_alloc(ptx::smem_addr(&ctl->tmem_base), Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    const uint64_t limit = a.wait_limit_ns;

    if (warp < 4) {
        // ------------------------------------------------------------ producers
        ptx::setmaxnreg_dec<PRODUCER_REGS>();
        const int row = threadIdx.x;  // 0..127
        const uint32_t row_off = (uint32_t)row * 128u;
        const uint32_t swz = (uint32_t)(row & 7);
        const int my_tiles = blockIdx.x < a.num_tiles ? (a.num_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        const int total = my_tiles * a.k_steps;
        LoadCursor cur;
        cursor_set_tile(cur, a, blockIdx.x, row);
        uint4 pf[PREFETCH][4];
#pragma unroll
        for (int d = 0; d < PREFETCH; ++d) {
            if (cur.tile < a.num_tiles) {
                cursor_load(cur, a, pf[d]);
                cursor_advance(cur, a, row);
            }
        }
        int stage = 0;
        uint32_t phase = 0;
        int b_tile = blockIdx.x, b_j = 0;  // filter block cursor (thread 0 only)
        int64_t b_issued = 0;
        bool ok = true;
        for (int it = 0; it < total && ok; it += PREFETCH) {
#pragma unroll
            for (int d = 0; d < PREFETCH; ++d) {
                if (it + d >= total) break;
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = pf[d][i];
                if (cur.tile < a.num_tiles) {  // keep PREFETCH items in flight
                    cursor_load(cur, a, pf[d]);
                    cursor_advance(cur, a, row);
                }
                if (!wait_phase(ptx::smem_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, limit, a.status)) {
                    ok = false;
                    break;
                }
                if (threadIdx.x == 0) {
                    const uint32_t bar = ptx::smem_addr(&ctl->b_full[stage]);
                    ptx::mbar_arrive_expect_tx(bar, B_BYTES);
                    const int nt = b_tile % a.n_tiles;
                    const uint8_t *src = a.wp + ((size_t)nt * a.k_steps + b_j) * (size_t)B_BYTES;
                    ptx::bulk_copy_g2s(b_smem + stage * B_BYTES, src, B_BYTES, bar);
                    ++b_issued;
                    if (++b_j == a.k_steps) {
                        b_j = 0;
                        b_tile += gridDim.x;
                    }
                }
                const uint32_t dst = a_smem + stage * A_BYTES + row_off;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 lo, hi;
                    cvt16(v[i], lo, hi);
                    ptx::st_shared_v4(dst + ((((uint32_t)(2 * i)) ^ swz) << 4), lo);
                    ptx::st_shared_v4(dst + ((((uint32_t)(2 * i + 1)) ^ swz) << 4), hi);
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->a_full[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (threadIdx.x == 0 && *abort_flag) {
            // let every filter copy this thread issued land before the CTA
            // exits: the newest copy into stage s completes phase
            // (copies into s) - 1 of b_full[s], and phases complete in order
            for (int s = 0; s < STAGES; ++s) {
                const int64_t n_s = b_issued / STAGES + (s < b_issued % STAGES ? 1 : 0);
                if (n_s > 0)
                    (void)drain_phase(ptx::smem_addr(&ctl->b_full[s]), (uint32_t)((n_s - 1) & 1), limit, a.status);
            }
        }
    } else if (warp < FIRST_EPI_WARP) {
        // ------------------------------------------------------------ MMA issuer
        ptx::setmaxnreg_dec<PRODUCER_REGS>();
        if (warp == MMA_WARP && lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(MT, NT);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t gi = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
                for (int g = 0; g < a.groups && ok; ++g) {
                    const int js = (int)(((int64_t)g * a.k_steps) / a.groups);
                    const int je = (int)(((int64_t)(g + 1) * a.k_steps) / a.groups);
                    const uint32_t slot = gi % NSLOT;
                    const uint32_t aph = (gi / NSLOT) & 1u;
                    if (!wait_phase(ptx::smem_addr(&ctl->acc_empty[slot]), aph ^ 1u, abort_flag, limit, a.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + slot * NT;
                    for (int j = js; j < je; ++j) {
                        if (!wait_phase(ptx::smem_addr(&ctl->a_full[stage]), phase, abort_flag, limit, a.status) ||
                            !wait_phase(ptx::smem_addr(&ctl->b_full[stage]), phase, abort_flag, limit, a.status)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint64_t adesc = ptx::smem_desc_sw128(a_smem + stage * A_BYTES);
                        const uint64_t bdesc = ptx::smem_desc_sw128(b_smem + stage * B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < KS / 16; ++kk) {
                            // advance 16 f16 = 32 bytes along K inside the swizzled row
                            ptx::mma_f16_ss(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                                            (j > js || kk > 0) ? 1u : 0u);
                        }
                        ptx::mma_commit(ptx::smem_addr(&ctl->empty[stage]));
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit(ptx::smem_addr(&ctl->acc_full[slot]));
                    ++gi;
                }
            }
            // all MMAs issued by this thread complete before tensor memory is freed
            ptx::mma_commit(ptx::smem_addr(&ctl->mma_done));
            (void)drain_phase(ptx::smem_addr(&ctl->mma_done), 0, limit, a.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        ptx::setmaxnreg_inc<EPILOGUE_REGS>();
        const int quad = warp & 3;                      // tensor-memory lanes this warp may access
        const int col0 = ((warp - FIRST_EPI_WARP) >> 2) * HALF;  // this warp's half of the columns
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)col0;
        uint32_t gi = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < a.num_tiles && ok; tile += gridDim.x) {
            const int mt = tile / a.n_tiles;
            const int nt = tile - mt * a.n_tiles;
            const int m = mt * MT + row;
            const bool valid = m < a.m_total;
            int64_t yoff = 0;
            if (valid) {
                const int pq = a.P * a.Q;
                const int n = m / pq;
                const int rem = m - n * pq;
                const int p = rem / a.Q;
                const int q = rem - p * a.Q;
                yoff = (int64_t)n * a.ys_n + (int64_t)p * a.ys_p + (int64_t)q * a.ys_q;
            }
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int g = 0; g < a.groups; ++g) {
                const uint32_t slot = gi % NSLOT;
                const uint32_t aph = (gi / NSLOT) & 1u;
                // tcgen05.ld is warp-collective: the whole warp proceeds or stops together
                const bool got = wait_phase(ptx::smem_addr(&ctl->acc_full[slot]), aph, abort_flag, limit, a.status);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < HALF / 32; ++cc) {
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(lane_base + slot * NT + cc * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[cc * 32 + i] += __float2int_rn(__uint_as_float(v[i]));
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->acc_empty[slot]));
                ++gi;
            }
            if (!ok) break;
            if (valid) {
                const int k0 = nt * NT + col0;
                int32_t *yrow = a.y + yoff;
#pragma unroll
                for (int c4 = 0; c4 < HALF / 4; ++c4) {
                    const int k = k0 + c4 * 4;
                    int32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        int32_t val = acc[c4 * 4 + e];
                        if (a.bias && k + e < a.K) val = (int32_t)((uint32_t)val + (uint32_t)__ldg(a.bias + k + e));
                        if (a.relu) val = max(val, 0);
                        o[e] = val;
                    }
                    if (a.y_vec && k + 3 < a.K) {
                        ptx::st_global_v4(yrow + (int64_t)k * a.ys_k, o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (k + e < a.K) yrow[(int64_t)(k + e) * a.ys_k] = o[e];
                    }
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == MMA_WARP) ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// ---------------------------------------------------------------- filter repack
// Writes B blocks: for n-tile nt and k-step j, NT rows (output channels) of
// 64 f16 (channels cb*64.. of tap (r, s) = divmod(j / c_steps, S), flipped for
// CONVOLUTION), each row's 16-byte chunk i stored at chunk position
// i ^ (row % 8): the image of the shared-memory stage, copied as one block.
__global__ void igemm_pack_filter_kernel(const int8_t *w, int64_t ws0, int64_t ws1, int64_t ws2, int64_t ws3,
                                         int32_t K, int32_t C, int32_t R, int32_t S, int32_t mode, int32_t c_steps,
                                         int32_t k_steps, int32_t n_tiles, int32_t nt_rows, uint8_t *wp) {
    const int64_t total = (int64_t)n_tiles * k_steps * nt_rows * 8;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int chunk = (int)(idx & 7);
        const int64_t t = idx >> 3;
        const int nl = (int)(t % nt_rows);
        const int64_t t2 = t / nt_rows;
        const int j = (int)(t2 % k_steps);
        const int nt = (int)(t2 / k_steps);
        const int k = nt * nt_rows + nl;
        const int tap = j / c_steps;
        const int cb = j - tap * c_steps;
        const int r = tap / S;
        const int s = tap - r * S;
        const int rf = mode ? R - 1 - r : r;
        const int sf = mode ? S - 1 - s : s;
        const int c0 = cb * KS + chunk * 8;
        uint32_t words[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            unsigned short hv[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int c = c0 + 2 * e + b;
                int v = 0;
                if (k < K && c < C)
                    v = w[(int64_t)k * ws0 + (int64_t)c * ws1 + (int64_t)rf * ws2 + (int64_t)sf * ws3];
                hv[b] = __half_as_ushort(__int2half_rn(v));
            }
            words[e] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
        }
        uint8_t *dst = wp + ((t2 * nt_rows + nl) * 128) + (((chunk ^ (nl & 7))) << 4);
        *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

// ---------------------------------------------------------------- image repack
// Channels-last copy of an image with arbitrary strides: xp[((n*H+h)*W+w)*c16 + c],
// channels C..c16-1 zero.  One thread writes 16 channels of one pixel; threads
// of a warp take neighbouring pixels so that reads along W coalesce for NCHW.
__global__ void igemm_pack_image_kernel(const int8_t *x, int64_t xs0, int64_t xs1, int64_t xs2, int64_t xs3,
                                        int64_t N, int32_t C, int32_t H, int32_t W, int32_t c16, int8_t *xp) {
    const int64_t pixels = N * H * W;
    const int cblocks = c16 / 16;
    const int64_t total = pixels * cblocks;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pix = idx % pixels;
        const int cb = (int)(idx / pixels);
        const int w = (int)(pix % W);
        const int64_t t = pix / W;
        const int h = (int)(t % H);
        const int64_t n = t / H;
        const int8_t *src = x + n * xs0 + (int64_t)h * xs2 + (int64_t)w * xs3;
        uint32_t words[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            uint32_t word = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int c = cb * 16 + e * 4 + b;
                const int8_t v = c < C ? __ldg(src + (int64_t)c * xs1) : (int8_t)0;
                word |= (uint32_t)(uint8_t)v << (8 * b);
            }
            words[e] = word;
        }
        *reinterpret_cast<uint4 *>(xp + pix * c16 + cb * 16) = make_uint4(words[0], words[1], words[2], words[3]);
    }
}

inline int64_t align256(int64_t v) { return (v + 255) & ~255LL; }

template <int NT>
conv_status launch_conv(const IgemmArgs &a, int grid, cudaStream_t st) {
    using Cfg = TileCfg<NT>;
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(igemm_conv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES) != cudaSuccess)
            return CONV_ERR_CUDA;
        attr_set[dev] = true;
    }
    igemm_conv_kernel<NT><<<grid, THREADS, Cfg::SMEM_BYTES, st>>>(a);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // namespace

bool igemm_supported(const ConvGeom &g) {
    const int64_t lim = (int64_t)1 << 30;
    if (g.H >= lim || g.W >= lim || g.P >= lim || g.Q >= lim) return false;
    if (g.pad_h >= (1 << 20) || g.pad_w >= (1 << 20) || g.str_h >= (1 << 20) || g.str_w >= (1 << 20) ||
        g.dil_h >= (1 << 20) || g.dil_w >= (1 << 20))
        return false;
    // largest image coordinate formed in the gather must stay in int32
    if ((g.P - 1) * g.str_h + (g.R - 1) * g.dil_h >= lim || (g.Q - 1) * g.str_w + (g.S - 1) * g.dil_w >= lim)
        return false;
    if (g.R * g.S > (1 << 20)) return false;
    return true;
}

void igemm_plan(const ConvGeom &g, const void *x_dev, IgemmPlan *pl) {
    const bool direct = g.xs[1] == 1 && (g.C % 16) == 0 && (g.xs[0] % 16) == 0 && (g.xs[2] % 16) == 0 &&
                        (g.xs[3] % 16) == 0 && (x_dev == nullptr || ((uintptr_t)x_dev % 16) == 0);
    pl->pack_x = !direct;
    pl->n_tile = g.K > 128 ? 256 : 128;
    pl->c16 = (g.C + 15) / 16 * 16;
    pl->c_steps = (g.C + KS - 1) / KS;
    pl->k_steps = g.R * g.S * pl->c_steps;
    pl->n_tiles = (g.K + pl->n_tile - 1) / pl->n_tile;
    pl->m_tiles = (g.N * g.P * g.Q + MT - 1) / MT;
    pl->wpack_bytes = (size_t)align256(pl->n_tiles * pl->k_steps * pl->n_tile * (int64_t)(KS * 2));
    pl->xpack_bytes = pl->pack_x ? (size_t)align256(g.N * g.H * g.W * pl->c16) : 0;
    pl->workspace_bytes = pl->wpack_bytes + pl->xpack_bytes;
}

conv_status igemm_pack_filter_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *w, void *workspace,
                                     void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    const int64_t total = pl.n_tiles * pl.k_steps * pl.n_tile * 8;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks == 0) return CONV_OK;
    igemm_pack_filter_kernel<<<(unsigned)blocks, 256, 0, st>>>(
        w, g.ws[0], g.ws[1], g.ws[2], g.ws[3], (int32_t)g.K, (int32_t)g.C, (int32_t)g.R, (int32_t)g.S, g.mode,
        (int32_t)pl.c_steps, (int32_t)pl.k_steps, (int32_t)pl.n_tiles, (int32_t)pl.n_tile, wp);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

conv_status igemm_main_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, int32_t *y,
                              const int32_t *bias, void *workspace, void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    IgemmArgs a;
    if (pl.pack_x) {
        int8_t *xp = reinterpret_cast<int8_t *>(wp + pl.wpack_bytes);
        const int64_t total = g.N * g.H * g.W * (pl.c16 / 16);
        int64_t blocks = (total + 255) / 256;
        if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
        igemm_pack_image_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, g.xs[0], g.xs[1], g.xs[2], g.xs[3], g.N,
                                                                  (int32_t)g.C, (int32_t)g.H, (int32_t)g.W,
                                                                  (int32_t)pl.c16, xp);
        if (cudaGetLastError() != cudaSuccess) return CONV_ERR_CUDA;
        a.x = xp;
        a.xs_n = g.H * g.W * pl.c16;
        a.xs_h = g.W * pl.c16;
        a.xs_w = pl.c16;
    } else {
        a.x = x;
        a.xs_n = g.xs[0];
        a.xs_h = g.xs[2];
        a.xs_w = g.xs[3];
    }
    a.wp = wp;
    a.y = y;
    a.bias = g.bias ? bias : nullptr;
    a.ys_n = g.ys[0]; a.ys_k = g.ys[1]; a.ys_p = g.ys[2]; a.ys_q = g.ys[3];
    a.H = (int32_t)g.H; a.W = (int32_t)g.W; a.P = (int32_t)g.P; a.Q = (int32_t)g.Q;
    a.K = (int32_t)g.K; a.S = (int32_t)g.S;
    a.c16 = (int32_t)pl.c16;
    a.c_steps = (int32_t)pl.c_steps;
    a.k_steps = (int32_t)pl.k_steps;
    a.groups = (int32_t)((pl.k_steps + MAX_GROUP_STEPS - 1) / MAX_GROUP_STEPS);
    a.pad_h = (int32_t)g.pad_h; a.pad_w = (int32_t)g.pad_w;
    a.str_h = (int32_t)g.str_h; a.str_w = (int32_t)g.str_w;
    a.dil_h = (int32_t)g.dil_h; a.dil_w = (int32_t)g.dil_w;
    a.m_total = (int32_t)(g.N * g.P * g.Q);
    a.n_tiles = (int32_t)pl.n_tiles;
    a.num_tiles = (int32_t)(pl.m_tiles * pl.n_tiles);
    a.relu = g.relu ? 1 : 0;
    a.y_vec = (g.ys[1] == 1 && (g.K % 4) == 0 && ((uintptr_t)y % 16) == 0 && (g.ys[0] % 4) == 0 &&
               (g.ys[2] % 4) == 0 && (g.ys[3] % 4) == 0)
                  ? 1
                  : 0;
    a.wait_limit_ns = wait_limit_ns();
    a.status = device_status_word();
    if (!a.status) return CONV_ERR_CUDA;
    if (a.num_tiles == 0) return CONV_OK;
    const int grid = a.num_tiles < sms ? a.num_tiles : sms;
    return pl.n_tile == 256 ? launch_conv<256>(a, grid, st) : launch_conv<128>(a, grid, st);
}

}  // namespace i8c
