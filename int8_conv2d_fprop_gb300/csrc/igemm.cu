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
// x NT output channels (NT = 128 for K <= 128, 192 for K <= 192, else 256).
// The image tile of a k-step is 128 output pixels x 64 channels of one tap.
// Kernel variants, chosen per call:
//  * NT = 256 (TMA): warp 5 lane 0 issues one TMA load per
//    k-step (an im2col box: window origins from the pixel order, the tap as
//    pixel offset, zeros outside the image; or, for an unpadded 1x1
//    stride-1 filter, a plain 2-D box of 128 pixel rows) into an int8
//    staging ring; warpgroup 0 converts each staged tile to f16 into the
//    128-byte-swizzled A stage in shared memory; warp 6 lane 0 brings the
//    matching pre-swizzled f16 filter block with one bulk async copy (or,
//    when the whole repacked filter fits in 128 KB, once per CTA: the
//    resident-filter variant).
//  * NT = 128 and NT = 192 (TMA): the same loads, issued by two warps (5
//    and 7) that own alternate staging slots; the converters write the f16
//    image tile into tensor memory (tcgen05.st) and the MMA reads A from
//    there (the tensor-memory-A form), which leaves shared memory to the
//    filter ring and the staging ring (NT = 128: six filter stages and eight
//    staging buffers; NT = 192: four and twelve); the 128-column epilogue
//    stores 32 columns per TMA store.
//  * NT = 128 and NT = 192 over an NCHW image (rows of at most 192 bytes,
//    stride 1 along W, tap offsets along W multiples of 4): the image is
//    read in place.  Each k-step loads, for every output row its tile's
//    pixels lie on, the whole image row of 64 channels (a 4-D TMA box
//    {W, 1, 64, 1}); the converters transpose while converting and write
//    tensor memory with tcgen05.st.16x256b, which permutes the tile's pixels
//    within each 32-lane quadrant (the epilogue follows) and the channels
//    within each 16 (the filter repack follows).
//  * NT = 128 and NT = 192 converting the filter (conv_fprop over a
//    channels-last image with a channel-contiguous filter): warp 6 lane 0
//    loads each k-step's int8 filter tile by TMA (a 4-D box {64, 1, 1, NT}
//    of the caller's filter) into a staging ring, and the converters write
//    it to the f16 filter stage next to their image tile: no repack launch.
//  * global loads (fallback when a TMA map cannot express the call):
//    warpgroup 0 threads each own one pixel row, gather 64 channels of one
//    tap with 16-byte loads one item ahead (address formed from stride,
//    padding and dilation), convert in registers and write the row; thread 0
//    also issues the filter block copies.
// In all, warp 4 allocates tensor memory and its lane 0 issues tcgen05.mma
// (M=128, N=NT, K=16 per instruction) into one of two accumulator slots:
//   warpgroups 2-3  epilogue, two warps per tensor-memory lane quadrant, each
//                owning NT/2 columns: tcgen05.ld each finished slot,
//                f32 -> int32, sum the groups, add bias, ReLU, optional int8
//                requantisation, TMA tensor stores (or plain stores).
// Work comes in units: whole tiles round by round, or runs of k-steps of cut
// tiles (few tiles with long reductions; a short partial last round) whose
// int32 sums igemm_split_reduce_kernel adds.
// Other images that are not channels-last with 16-byte channel runs are copied to
// channels-last first (igemm_pack_image_planes_kernel for NCHW planes,
// igemm_pack_image_kernel for any strides), keeping only the rows that
// the windows read when stride and dilation skip rows.
// Registers are moved from warpgroups 0-1 to the epilogue with setmaxnreg
// (the tensor-memory variants' converters keep 96, their issuers 64).
// Every wait is bounded in time; on expiry the CTA records
// CONV_ERR_DEVICE_TIMEOUT, stops, lets issued copies and MMAs finish and frees
// its tensor memory.
// Launch plans (tensor maps, grid, variant) are cached per call shape; a
// repeated call only re-targets the maps' addresses.  Behind the call's own
// filter repack the image issuers and converters start without waiting for
// it (griddepcontrol.wait only where the filter, the output or the workspace
// is touched).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <numeric>

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
// Tensor-memory variants: the converters (warpgroup 0) keep more registers,
// so that all of a k-step's shared loads are in flight at once, and the
// single-thread issuers of warpgroup 1 fewer.
constexpr int TMEM_CONV_REGS = 96;
constexpr int TMEM_ISSUE_REGS = 64;
static_assert(128 * TMEM_CONV_REGS + 128 * TMEM_ISSUE_REGS + 2 * 128 * EPILOGUE_REGS <= 65536,
              "register split exceeds the launch");
constexpr int PREFETCH = 1;  // register path: items in flight ahead of the one being stored
constexpr int STG_BYTES = MT * KS;  // one int8 im2col tile: 128 pixels x 64 channels
constexpr int A_ISSUER_WARP = 5;    // TMA path: issues the im2col loads
constexpr int A_ISSUER_WARP2 = 7;   // TMA path, image stages in tensor memory: second image-load issuer
constexpr int B_ISSUER_WARP = 6;    // TMA path: issues the filter block copies
// Output staging for TMA stores: per epilogue warp one or two buffers of 32
// rows x EPI_COLS int32 columns: 16 (64-byte rows, 64-byte swizzle) or, in
// the tensor-memory variant, 32 (128-byte rows, 128-byte swizzle: half as
// many store copies, which share each SM's TMA unit with the image loads).
// One buffer for 192- and 256-column tiles: a warp's next store then waits
// until its last one has read the buffer, which spaces the stores out
// between the main loop's loads (measured faster for those tiles; the
// 128-column tiles' short last epilogue wants two).
// Resident-filter variant: when the whole repacked filter of a call (one
// tile of output channels) fits in this many bytes, every CTA loads it once
// and keeps it in shared memory, so a k-step brings only its image tile.
constexpr int RESB_MAX_BYTES = 128 * 1024;
// Staging slot of the NCHW-row variants: the image rows a tile's 128 pixels
// lie on (up to 192 bytes of image row per channel), 64 channels each.
constexpr int NCHW_STG_BYTES = 192 * KS;
constexpr int NCHW_MAX_ROW_BYTES = NCHW_STG_BYTES / KS;

// kTma: the int8 image tile arrives by TMA (im2col mode) in a ring of
// STG_STAGES staging buffers and the producer warps convert it shared ->
// shared; otherwise the producer warps gather it with global loads.
// One ring of ST stages holds the f16 A tile (or, kTmemA, guards its
// tensor-memory stage) and the filter block of a k-step side by side,
// guarded by one "full" barrier (128 producer arrivals plus the filter
// copy's bytes) and one "empty" barrier (one MMA commit), so the single
// MMA-issuing thread waits once and commits once per k-step.  The int8
// staging ring of the TMA path (STG stages) runs ahead of it.
// Ring depths of the TMA path (tuning knobs; shared memory is the limit).
#ifndef IGEMM_ST_256
#define IGEMM_ST_256 3
#endif
#ifndef IGEMM_STG_256
#define IGEMM_STG_256 6
#endif
#ifndef IGEMM_ST_TM128
#define IGEMM_ST_TM128 6
#endif
#ifndef IGEMM_STG_TM128
#define IGEMM_STG_TM128 8
#endif
#ifndef IGEMM_ST_128
#define IGEMM_ST_128 4
#endif
#ifndef IGEMM_STG_128
#define IGEMM_STG_128 8
#endif

// kResB: the filter blocks of all k-steps stay resident (loaded once per
// CTA); the ring then holds image tiles only.
// kTmemA (128- and 192-column tiles, TMA path): the f16 image tile of a
// k-step goes to tensor memory (columns 2*NT.. next to the two accumulator
// slots, 32 columns per stage: 256..383 or 384..511) and the MMA reads it
// from there; the shared memory that held it goes to the filter ring and
// the int8 staging buffers (128 columns: six filter stages, eight staging
// buffers; 192 columns: four and twelve).
// kNchw (with kTmemA): the image is read in place from NCHW planes, each
// k-step's staging slot holding, for the rows its tile's pixels lie on,
// 64 channel rows of the whole image row (one 4-D TMA box per row); the
// converters transpose while converting (128 columns: five filter stages
// and six 12 KB staging slots; 192 columns: four and eight).
// kSelfB (with kTmemA, channels-last image): the kernel converts the filter
// itself.  Per k-step the filter issuer loads the int8 filter tile (NT
// output channels x 64 channels of one tap, a 4-D TMA box of the KRSC-like
// filter) into a staging ring, and the converters turn it into the f16
// filter stage beside the image tile: no repack launch (128 columns: six
// stages, eight image and four filter staging slots; 192 columns: four,
// six and four; 16 output columns per store).
template <int NT, bool kTma, bool kResB = false, bool kTmemA = false, bool kNchw = false, bool kSelfB = false>
struct TileCfg {
    static constexpr int B_BYTES = NT * KS * 2;
    static constexpr int STG_SLOT = kNchw ? NCHW_STG_BYTES : STG_BYTES;  // bytes per staging slot
    static constexpr int BSTG = kSelfB ? 4 : 0;                          // filter staging slots
    static constexpr int BSTG_SLOT = NT * KS;                            // int8 filter tile
    // (192-column tiles without kTmemA: 40 KB stages, four of them behind
    // four staging buffers)
    static constexpr int ST = kSelfB ? (NT == 128 ? 6 : 4)
                            : kNchw ? (NT == 128 ? 5 : 4)
                            : kTmemA ? (NT == 128 && !kResB ? IGEMM_ST_TM128 : 4)
                                     : (kResB ? 2 : (kTma ? (NT == 256 ? IGEMM_ST_256 : (NT == 192 ? 4 : IGEMM_ST_128))
                                                          : (NT == 128 ? 6 : 4)));
    static constexpr int STG_STAGES = kSelfB ? (NT == 128 ? 8 : 6)
                                    : kNchw ? (NT == 128 ? 6 : 8)
                                    : kTmemA ? (kResB ? 10 : (NT == 128 ? IGEMM_STG_TM128 : 12))
                                             : (kResB ? 6 : (kTma ? (NT == 256 ? IGEMM_STG_256 : (NT == 192 ? 4 : IGEMM_STG_128)) : 0));
    // output staging buffers per epilogue warp while the CTA has tiles to
    // come (one: each store waits for the last to have read it, which
    // spaces the stores out between the main loop's loads)
    static constexpr int EPI_BUFS = (kResB || NT >= 192) ? 1 : 2;
    // output columns per staged store: 32 for the 128-column tensor-memory
    // variant (its shared memory has room for 4 KB buffers), else 16
    static constexpr int EPI_COLS = (kTmemA && NT == 128 && !kSelfB) ? 32 : 16;
    static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 4;  // 2 or 4 KB
    static constexpr int A_SMEM = kTmemA ? 0 : ST * A_BYTES;
    static constexpr int B_AREA = kResB ? RESB_MAX_BYTES : ST * B_BYTES;
    static constexpr int SMEM_NO_EPI = 1024 /*align slack*/ + A_SMEM + B_AREA + STG_STAGES * STG_SLOT +
                                       BSTG * BSTG_SLOT + 1024 /*barriers*/;
    // buffers allocated: two where they fit, so that the CTA's last tile
    // (nothing left to overlap its stores with) alternates between them
    static constexpr int EPI_ALLOC = SMEM_NO_EPI + 8 * 2 * EPI_BUF_BYTES <= 227 * 1024 ? 2 : EPI_BUFS;
    static constexpr int EPI_BYTES = 8 * EPI_ALLOC * EPI_BUF_BYTES;
    // (allocations are powers of two: two 192-column slots take 512)
    static constexpr int TMEM_COLS = (kTmemA || NT == 192) ? 512 : NSLOT * NT;
    static constexpr int TMEM_A_COL = NSLOT * NT;  // kTmemA: first column of the image stages
    // Warps that issue the image loads (kTmemA: warps 5 and 7, one thread
    // each): issuer i issues the loads into the staging slots s % A_ISSUERS
    // == i.  Issuing a TMA load takes its thread a few hundred ns, so one
    // issuer keeps only about four loads in flight; the 128-column tiles
    // stream their image from HBM and need more.  (Lanes of one warp would
    // not help: their divergent branches run one after the other.)
    static constexpr int A_ISSUERS = kTmemA ? 2 : 1;
    static_assert(STG_STAGES % A_ISSUERS == 0, "staging slots split evenly between the issuers");
    static constexpr int SMEM_BYTES = SMEM_NO_EPI + EPI_BYTES;
    static_assert(!kResB || kTma, "the resident filter needs the TMA producers");
    static_assert(!kNchw || (kTmemA && !kResB), "NCHW rows feed the tensor-memory image stages");
    static_assert(!kSelfB || (kTmemA && !kResB && !kNchw), "in-kernel filter conversion: tensor-memory variants");
    static_assert(!kTmemA || (kTma && NT <= 192 && TMEM_A_COL + ST * 32 <= 512), "image stages in tensor memory");
    static_assert(TMEM_COLS <= 512, "tensor memory has 512 columns");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(ST <= 8 && STG_STAGES <= 16, "the control block has 8 ring and 16 staging barriers");
};

// Slot index and phase parity of a ring of N mbarrier-guarded buffers.
template <int N>
struct Ring {
    int idx = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next() {
        if (++idx == N) {
            idx = 0;
            phase ^= 1u;
        }
    }
};

// One work unit: a tile and its run [kb, ke) of k-steps; split >= 0 for a
// run of a tile that several CTAs share.
struct Unit {
    int tile, kb, ke, split;
};

__device__ __forceinline__ Unit unit_at(int u, int full_units, int splits, int k_steps) {
    Unit w;
    if (u < full_units) {
        w.tile = u;
        w.kb = 0;
        w.ke = k_steps;
        w.split = -1;
    } else {
        const int t = u - full_units;
        w.tile = full_units + t / splits;
        w.split = t - (t / splits) * splits;
        w.kb = (int)(((int64_t)w.split * k_steps) / splits);
        w.ke = (int)(((int64_t)(w.split + 1) * k_steps) / splits);
    }
    return w;
}

// Groups of a run of kn k-steps: the fewest runs of at most MAX_GROUP_STEPS
// (group g covers k-steps g*kn/ng .. (g+1)*kn/ng - 1 of the run).
__device__ __forceinline__ int groups_of(int kn) { return (kn + MAX_GROUP_STEPS - 1) / MAX_GROUP_STEPS; }

// floor(n / d) for 0 <= n < 2^31 and 1 <= d < 2^31 by one multiply-high and
// a shift: division by an invariant integer (Granlund and Montgomery, PLDI
// 1994).  With l = ceil(log2 d) and m = ceil(2^(31+l) / d) = (2^(31+l) + e) / d,
// 0 <= e < d, the quotient n*m / 2^(31+l) exceeds n/d by n*e / (d*2^(31+l)),
// which is below 1/d because n*e < 2^31 * 2^l: both have the same floor.
// d > 2^(l-1) keeps m below 2^32, and the floor is umulhi(n, m) >> (l - 1).
// m == 0 stands for d == 1.  The issuers set up each unit's coordinates with
// these instead of runtime divisions, which cost them about a microsecond per
// unit while the other warps poll.
struct FastDiv {
    uint32_t m, s;
};

__device__ __forceinline__ int fdiv(int n, FastDiv f) {
    return f.m ? (int)(__umulhi((uint32_t)n, f.m) >> f.s) : n;
}

inline FastDiv make_fastdiv(int64_t d) {
    FastDiv f = {0u, 0u};
    if (d <= 1) return f;
    int l = 0;
    while ((1ll << l) < d) ++l;
    const uint64_t two_p = 1ull << (31 + l);
    f.m = (uint32_t)((two_p + (uint64_t)d - 1) / (uint64_t)d);
    f.s = (uint32_t)(l - 1);
    return f;
}

struct IgemmArgs {
    CUtensorMap tmap_x;  // im2col map of the channels-last image, or its 2-D pixel-row map (TMA path only)
    CUtensorMap tmap_y;  // output map: 2-D [pixels][K] (y_tma 1) or 3-D [N][K][P*Q] (y_tma 2)
    CUtensorMap tmap_w;  // kSelfB: 4-D {C, S, R, K} map of the int8 filter
    const int8_t *x;     // channels-last image
    const uint8_t *wp;   // repacked f16 filter blocks
    void *y;             // int32 output, or int8 when out_int8
    int32_t out_int8, out_shift;
    const int32_t *bias;
    int64_t xs_n, xs_h, xs_w;  // element (= byte) strides of the channels-last image
    int64_t ys_n, ys_k, ys_p, ys_q;
    int32_t H, W, P, Q, K, R, S;
    int32_t mode;        // CONVOLUTION: filter taps flipped (kSelfB reads the filter itself)
    int32_t c16;         // channel bytes per pixel that may be loaded (multiple of 16)
    int32_t c_steps, k_steps;
    int32_t pad_h, pad_w, str_h, str_w, dil_h, dil_w;
    int32_t m_total, n_tiles, num_tiles;
    // Work units.  Units below full_units are whole tiles (unit u = tile u).
    // The tiles from full_units on (all of them when there are fewer tiles
    // than SMs and long reductions; a short partial last round otherwise)
    // are cut into `splits` runs of k-steps: unit full_units + t covers run
    // t % splits of tile full_units + t / splits, and writes its raw int32
    // sums to tail_part for the reduction kernel.
    int32_t full_units, splits, num_units;
    int32_t *tail_part;  // [cut tile][split][MT rows][NT columns]
    int32_t relu, y_vec;
    int32_t a_rows;      // TMA path: 1x1, stride 1, no padding: the image tile is a plain 2-D box of
                         // pixel rows (output pixel m reads image pixel m)
    int32_t y_tma;       // TMA stores: 1 pixel-major with contiguous channels, 2 channel-major
                         // (each channel's P*Q pixels contiguous, P*Q a multiple of 32)
    FastDiv fd_nt, fd_pq, fd_q, fd_cs, fd_s;  // by n_tiles, P*Q, Q, c_steps, S
    // 1: launched right behind this call's own filter repack (an ordinary
    // launch, so every earlier kernel of the stream had completed when it
    // started): the image is final, and the TMA image loads need not wait
    // for the repack to finish (only the filter copies do)
    int32_t early_image;
    uint64_t wait_limit_ns;
    int *status;         // device status word
};

struct SharedCtl {
    uint64_t full[8], empty[8];          // A + filter ring
    uint64_t stg_full[16], stg_empty[16];  // TMA path: im2col tile landed / converted
    uint64_t bstg_full[8], bstg_empty[8];  // kSelfB: int8 filter tile landed / converted
    uint64_t acc_full[NSLOT];
    uint64_t acc_empty[NSLOT];
    uint64_t mma_done;
    uint64_t b_res;                      // resident filter landed (kResB)
    uint32_t tmem_base;
    int32_t abort_flag;
};
static_assert(sizeof(SharedCtl) <= 1024, "control block too large");

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or
// the time limit passed (then the CTA is marked aborting and the device status
// word records the timeout).  backoff_ns > 0: sleep that long between polls,
// for waits off the k-step critical path (an epilogue warp waiting for its
// next tile, an issuer waiting for a free slot), so that polling does not take
// issue slots from the converters and the MMA thread on the same scheduler.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int32_t *abort_flag,
                                           uint64_t limit_ns, int *status, uint32_t backoff_ns = 0) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    while (true) {
        if (backoff_ns) {
#pragma unroll 1
            for (int i = 0; i < 8; ++i) {
                __nanosleep(backoff_ns);
                if (ptx::mbar_try_wait(bar, parity)) return true;
            }
        } else {
            // on the k-step critical path: poll without suspending (a
            // suspended try_wait resumes some time after the phase completes)
#pragma unroll 1
            for (int i = 0; i < 64; ++i)
                if (ptx::mbar_test_wait(bar, parity)) return true;
        }
        if (*abort_flag) return false;
        if (ptx::global_timer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            atomicExch(status, (int)CONV_ERR_DEVICE_TIMEOUT);
            return false;
        }
    }
}

constexpr uint32_t kIssuerBackoffNs = 32;    // image / filter issuers waiting for a free slot
constexpr uint32_t kEpilogueBackoffNs = 128; // epilogue warps waiting for a finished accumulator

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

// Where one producer thread is in its (unit, k-step) sequence.
struct LoadCursor {
    int u;          // work unit, >= num_units when done
    int j, je;      // current and end k-step of the unit
    int cb, r, s;   // channel block and tap of k-step j
    int64_t xoff;   // n * xs_n
    int h0, w0;
    bool valid;     // this thread's pixel row exists
};

__device__ __forceinline__ void cursor_set_unit(LoadCursor &c, const IgemmArgs &a, int u, int row) {
    c.u = u;
    const Unit w = unit_at(u < a.num_units ? u : 0, a.full_units, a.splits, a.k_steps);
    c.j = w.kb;
    c.je = w.ke;
    const int tap = w.kb / a.c_steps;
    c.cb = w.kb - tap * a.c_steps;
    c.r = tap / a.S;
    c.s = tap - c.r * a.S;
    const int mt = w.tile / a.n_tiles;
    const int m = mt * MT + row;
    c.valid = u < a.num_units && m < a.m_total;
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

__device__ __forceinline__ void cursor_advance(LoadCursor &c, const IgemmArgs &a, int row, int gdim) {
    if (++c.j == c.je) {
        cursor_set_unit(c, a, c.u + gdim, row);
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

// Lets every copy issued into a ring of `depth` slots land: the newest copy
// into slot s completes phase (copies into s) - 1, and phases complete in
// order.  Used only after an abort.  drain_ring_owned: the same for the
// slots s % lanes == lane of a ring walked up to position `stop`, whose
// copies that lane issued.  A filter copy shares its "full" barrier
// with the 128 producer arrivals, which an aborting CTA may never make; the
// wait is then cut off after DRAIN_LIMIT_NS.  Copies issued before the abort
// (itself a wait that ran out after the full time limit) have long landed.
constexpr uint64_t DRAIN_LIMIT_NS = 10000000;  // 10 ms
__device__ __forceinline__ void drain_ring(uint64_t *bars, int depth, int64_t issued, uint64_t limit, int *status) {
    for (int s = 0; s < depth; ++s) {
        const int64_t n_s = issued / depth + (s < issued % depth ? 1 : 0);
        if (n_s > 0) (void)drain_phase(ptx::smem_addr(&bars[s]), (uint32_t)((n_s - 1) & 1), limit, status);
    }
}

__device__ __forceinline__ void drain_ring_owned(uint64_t *bars, int depth, int64_t stop, int lane, int lanes,
                                                 uint64_t limit, int *status) {
    for (int s = lane; s < depth; s += lanes) {
        const int64_t n_s = stop / depth + (s < stop % depth ? 1 : 0);
        if (n_s > 0) (void)drain_phase(ptx::smem_addr(&bars[s]), (uint32_t)((n_s - 1) & 1), limit, status);
    }
}

// L2 prefetch of the image tiles of this CTA's first `depth` k-steps (the
// loads the image issuers start with), issued before the kernel waits for
// the grids it depends on: L2 is the GPU's point of coherence, so a line
// fetched early is still updated by any earlier kernel's writes, and the
// loads themselves come after the wait.
template <bool kNchw>
__device__ __forceinline__ void prefetch_first_image_tiles(const IgemmArgs &a, int bid, int depth) {
    if (bid >= a.num_units) return;
    const Unit wu = unit_at(bid, a.full_units, a.splits, a.k_steps);
    const int pq = a.P * a.Q;
    const int m0 = fdiv(wu.tile, a.fd_nt) * MT;
    const int n0 = fdiv(m0, a.fd_pq);
    const int rem = m0 - n0 * pq;
    const int p0 = fdiv(rem, a.fd_q);
    const int q0 = rem - p0 * a.Q;
    const int nrows = kNchw ? fdiv(q0 + MT - 1, a.fd_q) + 1 : 1;
    const int tap = fdiv(wu.kb, a.fd_cs);
    int cb = wu.kb - tap * a.c_steps;
    int r = fdiv(tap, a.fd_s);
    int s = tap - r * a.S;
    const int n = wu.ke - wu.kb < depth ? wu.ke - wu.kb : depth;
#pragma unroll 1
    for (int j = 0; j < n; ++j) {
        if (kNchw) {
            int pb = p0, nb = n0;
#pragma unroll 1
            for (int b = 0; b < nrows; ++b) {
                ptx::tma_prefetch_4d(&a.tmap_x, 0, pb * a.str_h - a.pad_h + r * a.dil_h, cb * KS, nb);
                if (++pb == a.P) {
                    pb = 0;
                    ++nb;
                }
            }
        } else if (a.a_rows) {
            ptx::tma_prefetch_2d(&a.tmap_x, cb * KS, m0);
        } else {
            ptx::tma_prefetch_im2col_4d(&a.tmap_x, cb * KS, q0 * a.str_w - a.pad_w, p0 * a.str_h - a.pad_h, n0,
                                        (uint16_t)(s * a.dil_w), (uint16_t)(r * a.dil_h));
        }
        if (++cb == a.c_steps) {
            cb = 0;
            if (++s == a.S) {
                s = 0;
                ++r;
            }
        }
    }
}

// The kernel's body for one CTA: `a` holds the call's arguments, bid is the
// CTA's index among the gdim CTAs that share the call's work units.
template <int NT, bool kTma, bool kResB, bool kTmemA, bool kNchw, bool kSelfB>
__device__ __forceinline__ void conv_cta(const IgemmArgs &a, const int bid, const int gdim) {
    using Cfg = TileCfg<NT, kTma, kResB, kTmemA, kNchw, kSelfB>;
    constexpr int STG_SLOT = Cfg::STG_SLOT;
    constexpr int ST = Cfg::ST;
    constexpr int STG = Cfg::STG_STAGES;
    constexpr int B_BYTES = Cfg::B_BYTES;
    constexpr int HALF = NT / 2;  // columns per epilogue thread
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_addr(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t *const base_ptr = smem_raw + (base - raw_addr);
    const uint32_t a_smem = base;
    const uint32_t b_smem = a_smem + Cfg::A_SMEM;
    const uint32_t stg_smem = b_smem + Cfg::B_AREA;
    const uint32_t bstg_smem = stg_smem + STG * STG_SLOT;
    const uint32_t epi_smem = bstg_smem + Cfg::BSTG * Cfg::BSTG_SLOT;
    SharedCtl *ctl = reinterpret_cast<SharedCtl *>(base_ptr + Cfg::A_SMEM + Cfg::B_AREA + STG * STG_SLOT +
                                                   Cfg::BSTG * Cfg::BSTG_SLOT + Cfg::EPI_BYTES);
    volatile int32_t *abort_flag = &ctl->abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int total = 0;  // k-steps of all units of this CTA
    for (int u = bid; u < a.num_units; u += gdim) {
        const Unit w = unit_at(u, a.full_units, a.splits, a.k_steps);
        total += w.ke - w.kb;
    }
    // (every CTA walks a tile's reduction in k-step order, so at any moment
    // most SMs read the same filter block: faster, from L2, than spreading
    // them over the blocks by starting each CTA at its own k-step)

    if (threadIdx.x == 0) {
        for (int i = 0; i < ST; ++i) {
            // 128 producer arrivals (A tile written) + 1 arrival with the
            // filter copy's byte count (no filter copy per k-step when the
            // filter is resident or the converters write the filter stage)
            ptx::mbar_init(ptx::smem_addr(&ctl->full[i]), (kResB || kSelfB) ? 128 : 129);
            ptx::mbar_init(ptx::smem_addr(&ctl->empty[i]), 1);
        }
        ptx::mbar_init(ptx::smem_addr(&ctl->b_res), 1);
        for (int i = 0; i < STG; ++i) {
            ptx::mbar_init(ptx::smem_addr(&ctl->stg_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->stg_empty[i]), 128);
        }
        for (int i = 0; i < Cfg::BSTG; ++i) {
            ptx::mbar_init(ptx::smem_addr(&ctl->bstg_full[i]), 1);
            ptx::mbar_init(ptx::smem_addr(&ctl->bstg_empty[i]), 128);
        }
        if (kTma) ptx::prefetch_tensormap(&a.tmap_x);
        if (kSelfB) ptx::prefetch_tensormap(&a.tmap_w);
        if (a.y_tma) ptx::prefetch_tensormap(&a.tmap_y);
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
    // launched as a programmatic dependent of the filter (or image) repack:
    // the set-up above overlaps its tail, nothing below runs before its
    // writes are visible.  Without cut tiles, a programmatic dependent that
    // follows (the next call's convolution) may be scheduled from here on; it
    // waits for this grid before touching memory.  (With cut tiles the
    // reduction follows, and it starts when this grid ends, so that the next
    // convolution's CTAs cannot take SMs from it.)
    // (behind this call's own filter repack, the image-load issuers and the
    // converters, which touch no global memory, start at once)
    const bool image_role = warp < 4 || warp == A_ISSUER_WARP || warp == A_ISSUER_WARP2;
    // (otherwise, in the 128- and 192-column variants, the first image tiles
    // are brought into L2 while the wait lasts, by an epilogue warp, which
    // has nothing to do until then, so that the image issuers' loads do not
    // queue behind the prefetches.  Not in calls that cut tiles: a call like
    // them follows its reduction kernel, which lets nothing start early, so
    // there is no wait to fill.  The 256-column kernel, measured slower with
    // the prefetch compiled in, does without.)
    if (kTma && kTmemA && !a.early_image && a.splits <= 1 && warp == FIRST_EPI_WARP && lane == 0)
        prefetch_first_image_tiles<kNchw>(a, bid, STG);
    if (!(kTma && a.early_image && image_role)) ptx::grid_dependency_wait();
    if (a.splits <= 1) ptx::launch_dependents();

    if (warp < 4 && kNchw) {
        // ---------------------------------------- converters (NCHW rows to tensor memory)
        // The staged slot holds, for each output row the tile's pixels lie
        // on (box b), 64 channel rows of the whole image row (W bytes each).
        // With stride 1 along W and tap offsets s*dil_w - pre_w that are
        // multiples of 4, the tile's pixels 4t .. 4t+3 are four consecutive
        // bytes of every channel row.  Thread (j, u) = (lane / 4, lane % 4)
        // of warp w takes pixels 32w + 4j .. +3 and channels 16i + u + 4v
        // (i, v = 0..3): sixteen 4-byte loads (the four u read four
        // neighbouring channel rows).  A 4x4 byte transpose inside the
        // conversion gives each pixel its channels, and tcgen05.st.16x256b
        // writes them: in the warp's first 16 lanes, lane j holds pixel 4j
        // and lane j+8 pixel 4j+1; in the second, lanes 16+j and 24+j hold
        // pixels 4j+2 and 4j+3 (lane l of the quadrant: pixel
        // 4*(l%8) + l/8, which the epilogue follows).  Column 8i + 2u holds
        // channels 16i + u and 16i + u + 4, column 8i + 2u + 1 channels
        // 16i + u + 8 and 16i + u + 12: within each 16 channels the K order
        // swaps the two 2-bit digits of the channel index, and the filter
        // repack writes the filter blocks in the same order.
        ptx::setmaxnreg_dec<TMEM_CONV_REGS>();
        const int jq = lane >> 2, u = lane & 3;
        const uint32_t lanes_lo = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)Cfg::TMEM_A_COL;
        const uint32_t lanes_hi = lanes_lo + (16u << 16);
        const uint32_t rowb = (uint32_t)a.W;          // bytes per channel row
        const uint32_t boxb = (uint32_t)(KS * a.W);   // bytes per image-row box
        const int pq = a.P * a.Q;
        Ring<ST> ra;
        Ring<STG> rs;
        bool ok = true;
        for (int uu = bid; uu < a.num_units && ok; uu += gdim) {
            const Unit wu = unit_at(uu, a.full_units, a.splits, a.k_steps);
            const int kn = wu.ke - wu.kb;
            const int m0 = fdiv(wu.tile, a.fd_nt) * MT;
            const int rem = m0 - fdiv(m0, a.fd_pq) * pq;
            const int q0 = rem - fdiv(rem, a.fd_q) * a.Q;
            // this thread's pixels in the run of output rows that starts at
            // the tile's first pixel: row b, column q
            const int f = q0 + warp * 32 + jq * 4;
            const int b = fdiv(f, a.fd_q);
            const int q = f - b * a.Q;
            const uint32_t pix = (uint32_t)b * boxb + (uint32_t)u * rowb;
            // the unit's k-steps in order, for the tap column s
            const int tap = fdiv(wu.kb, a.fd_cs);
            int cb = wu.kb - tap * a.c_steps;
            int r = fdiv(tap, a.fd_s);
            int s = tap - r * a.S;
#pragma unroll 1
            for (int j = 0; j < kn; ++j) {
                bool got = wait_phase(ptx::smem_addr(&ctl->stg_full[rs.idx]), rs.phase, abort_flag, limit, a.status);
                got = got && wait_phase(ptx::smem_addr(&ctl->empty[ra.idx]), ra.phase ^ 1u, abort_flag, limit, a.status);
                // tcgen05.st is warp-collective: the whole warp proceeds or stops together
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                const int wpos = q + s * a.dil_w - a.pad_w;
                const bool inb = (unsigned)wpos < (unsigned)a.W;  // all four pixels in or all out
                const uint32_t src = stg_smem + rs.idx * STG_SLOT + pix + (uint32_t)wpos;
                uint32_t xw[16];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        xw[4 * i + v] = inb ? ptx::ld_shared_b32(src + (uint32_t)(16 * i + 4 * v) * rowb) : 0u;
                // gl[2i], gl[2i+1]: bytes [x0.b0, x1.b0, x0.b1, x1.b1] of the words
                // of channels (16i + u, +4) and (+8, +12), i.e. those channels of
                // pixels 4j and 4j+1; gh likewise bytes 2 and 3, pixels 4j+2, 4j+3
                uint32_t gl[8], gh[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t x0 = xw[2 * i] ^ 0x80808080u, x1 = xw[2 * i + 1] ^ 0x80808080u;
                    gl[i] = __byte_perm(x0, x1, 0x5140);
                    gh[i] = __byte_perm(x0, x1, 0x7362);
                }
                uint32_t v[16];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[4 * i + 0] = cvt_pair(gl[2 * i], 0x4140);      // lane j:      pixel 4j
                    v[4 * i + 1] = cvt_pair(gl[2 * i + 1], 0x4140);
                    v[4 * i + 2] = cvt_pair(gl[2 * i], 0x4342);      // lane j + 8:  pixel 4j + 1
                    v[4 * i + 3] = cvt_pair(gl[2 * i + 1], 0x4342);
                }
                ptx::tmem_st_16x256b_x4(lanes_lo + (uint32_t)(ra.idx * 32), v);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[4 * i + 0] = cvt_pair(gh[2 * i], 0x4140);      // lane 16 + j: pixel 4j + 2
                    v[4 * i + 1] = cvt_pair(gh[2 * i + 1], 0x4140);
                    v[4 * i + 2] = cvt_pair(gh[2 * i], 0x4342);      // lane 24 + j: pixel 4j + 3
                    v[4 * i + 3] = cvt_pair(gh[2 * i + 1], 0x4342);
                }
                ptx::tmem_st_16x256b_x4(lanes_hi + (uint32_t)(ra.idx * 32), v);
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->stg_empty[rs.idx]));
                ptx::mbar_arrive(ptx::smem_addr(&ctl->full[ra.idx]));
                ra.next();
                rs.next();
                if (++cb == a.c_steps) {
                    cb = 0;
                    if (++s == a.S) {
                        s = 0;
                        ++r;
                    }
                }
            }
        }
    } else if (warp < 4 && kTmemA) {
        // ------------------------------------------------- converters (to tensor memory)
        // Thread t converts pixel row t of the staged tile (its 64 channel
        // bytes, 16-byte chunk c stored at chunk position c ^ ((t >> 1) & 3)
        // by the TMA 64-byte swizzle: each 8 rows cover all banks) and writes
        // the 32 f16 pairs to tensor-memory lane t (warp w owns lanes
        // 32w..32w+31), column j holding channels 2j and 2j+1.
        // kSelfB: the same threads also convert the k-step's int8 filter
        // tile (NT rows of 64 bytes in its staging slot) into the f16 filter
        // stage of the ring, four neighbouring lanes per row and 128-byte
        // swizzled rows (the layout of a repacked block), while the tensor
        // memory store of the image tile completes.
        ptx::setmaxnreg_dec<TMEM_CONV_REGS>();
        const int row = threadIdx.x;
        const uint32_t sw = (uint32_t)((row >> 1) & 3);
        const uint32_t lane_col0 = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)Cfg::TMEM_A_COL;
        const uint32_t bchunk = threadIdx.x & 3u;
        Ring<ST> ra;
        Ring<STG> rs;
        Ring<(Cfg::BSTG > 0 ? Cfg::BSTG : 1)> rb;
        for (int it = 0; it < total; ++it) {
            bool got = wait_phase(ptx::smem_addr(&ctl->stg_full[rs.idx]), rs.phase, abort_flag, limit, a.status);
            got = got && wait_phase(ptx::smem_addr(&ctl->empty[ra.idx]), ra.phase ^ 1u, abort_flag, limit, a.status);
            if (kSelfB)
                got = got && wait_phase(ptx::smem_addr(&ctl->bstg_full[rb.idx]), rb.phase, abort_flag, limit, a.status);
            // tcgen05.st is warp-collective: the whole warp proceeds or stops together
            if (!__all_sync(0xffffffffu, got)) break;
            const uint32_t src = stg_smem + rs.idx * STG_SLOT + (uint32_t)row * 64u;
            uint4 vin[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) vin[c] = ptx::ld_shared_v4(src + ((((uint32_t)c) ^ sw) << 4));
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint4 lo, hi;
                cvt16(vin[c], lo, hi);
                w[8 * c + 0] = lo.x; w[8 * c + 1] = lo.y; w[8 * c + 2] = lo.z; w[8 * c + 3] = lo.w;
                w[8 * c + 4] = hi.x; w[8 * c + 5] = hi.y; w[8 * c + 6] = hi.z; w[8 * c + 7] = hi.w;
            }
            ptx::tmem_st_32x32b_x32(lane_col0 + (uint32_t)(ra.idx * 32), w);
            if (kSelfB) {
                const uint32_t bsrc = bstg_smem + rb.idx * Cfg::BSTG_SLOT + bchunk * 16u;
                const uint32_t bdst = b_smem + ra.idx * B_BYTES;
                uint4 vb[NT / 32];
#pragma unroll
                for (int i = 0; i < NT / 32; ++i)
                    vb[i] = ptx::ld_shared_v4(bsrc + (uint32_t)((threadIdx.x >> 2) + 32 * i) * 64u);
#pragma unroll
                for (int i = 0; i < NT / 32; ++i) {
                    const uint32_t brow = (uint32_t)((threadIdx.x >> 2) + 32 * i);
                    uint4 lo, hi;
                    cvt16(vb[i], lo, hi);
                    const uint32_t rdst = bdst + brow * 128u;
                    const uint32_t swz = brow & 7u;
                    ptx::st_shared_v4(rdst + (((2u * bchunk) ^ swz) << 4), lo);
                    ptx::st_shared_v4(rdst + (((2u * bchunk + 1u) ^ swz) << 4), hi);
                }
                // the filter stage is read by the tensor core (async proxy)
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->bstg_empty[rb.idx]));
                rb.next();
            }
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(ptx::smem_addr(&ctl->stg_empty[rs.idx]));
            ptx::mbar_arrive(ptx::smem_addr(&ctl->full[ra.idx]));
            ra.next();
            rs.next();
        }
    } else if (warp < 4 && kTma) {
        // ------------------------------------------------------------ converters
        // The im2col tile in staging holds pixel row i at i*64 bytes.  Four
        // neighbouring lanes take the four 16-byte chunks of one row, so a
        // warp reads 8 whole rows per instruction and writes them to the
        // swizzled f16 stage without bank conflicts.  A thread's four loads
        // go out together before any conversion waits on one.
        ptx::setmaxnreg_dec<PRODUCER_REGS>();
        const uint32_t chunk = threadIdx.x & 3;
        const int row0 = (warp << 5) + (lane >> 2);
        Ring<ST> ra;
        Ring<STG> rs;
        for (int it = 0; it < total; ++it) {
            if (!wait_phase(ptx::smem_addr(&ctl->stg_full[rs.idx]), rs.phase, abort_flag, limit, a.status)) break;
            if (!wait_phase(ptx::smem_addr(&ctl->empty[ra.idx]), ra.phase ^ 1u, abort_flag, limit, a.status))
                break;
            const uint32_t src = stg_smem + rs.idx * STG_SLOT + chunk * 16u;
            const uint32_t dst = a_smem + ra.idx * A_BYTES;
            uint4 vin[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) vin[i] = ptx::ld_shared_v4(src + (uint32_t)(row0 + 8 * i) * 64u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t row = (uint32_t)(row0 + 8 * i);
                uint4 lo, hi;
                cvt16(vin[i], lo, hi);
                const uint32_t rdst = dst + row * 128u;
                const uint32_t swz = row & 7u;
                ptx::st_shared_v4(rdst + (((2u * chunk) ^ swz) << 4), lo);
                ptx::st_shared_v4(rdst + (((2u * chunk + 1u) ^ swz) << 4), hi);
            }
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(ptx::smem_addr(&ctl->stg_empty[rs.idx]));
            ptx::mbar_arrive(ptx::smem_addr(&ctl->full[ra.idx]));
            ra.next();
            rs.next();
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ producers
        ptx::setmaxnreg_dec<PRODUCER_REGS>();
        const int row = threadIdx.x;  // 0..127
        const uint32_t row_off = (uint32_t)row * 128u;
        const uint32_t swz = (uint32_t)(row & 7);
        LoadCursor cur;
        cursor_set_unit(cur, a, bid, row);
        uint4 pf[PREFETCH][4];
#pragma unroll
        for (int d = 0; d < PREFETCH; ++d) {
            if (cur.u < a.num_units) {
                cursor_load(cur, a, pf[d]);
                cursor_advance(cur, a, row, gdim);
            }
        }
        Ring<ST> rg;
        // filter block cursor (thread 0 only): unit b_u, k-step b_j < b_je
        int b_u = bid;
        Unit bw = unit_at(b_u < a.num_units ? b_u : 0, a.full_units, a.splits, a.k_steps);
        int b_j = bw.kb, b_je = bw.ke;
        int64_t b_issued = 0;
        bool ok = true;
        for (int it = 0; it < total && ok; it += PREFETCH) {
#pragma unroll
            for (int d = 0; d < PREFETCH; ++d) {
                if (it + d >= total) break;
                uint4 v[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = pf[d][i];
                if (cur.u < a.num_units) {  // keep PREFETCH items in flight
                    cursor_load(cur, a, pf[d]);
                    cursor_advance(cur, a, row, gdim);
                }
                if (!wait_phase(ptx::smem_addr(&ctl->empty[rg.idx]), rg.phase ^ 1u, abort_flag, limit, a.status)) {
                    ok = false;
                    break;
                }
                if (threadIdx.x == 0) {
                    const uint32_t bar = ptx::smem_addr(&ctl->full[rg.idx]);
                    ptx::mbar_arrive_expect_tx(bar, B_BYTES);
                    const int nt = bw.tile % a.n_tiles;
                    const uint8_t *src = a.wp + ((size_t)nt * a.k_steps + b_j) * (size_t)B_BYTES;
                    ptx::bulk_copy_g2s(b_smem + rg.idx * B_BYTES, src, B_BYTES, bar);
                    ++b_issued;
                    if (++b_j == b_je) {
                        b_u += gdim;
                        bw = unit_at(b_u < a.num_units ? b_u : 0, a.full_units, a.splits, a.k_steps);
                        b_j = bw.kb;
                        b_je = bw.ke;
                    }
                }
                const uint32_t dst = a_smem + rg.idx * A_BYTES + row_off;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint4 lo, hi;
                    cvt16(v[i], lo, hi);
                    ptx::st_shared_v4(dst + ((((uint32_t)(2 * i)) ^ swz) << 4), lo);
                    ptx::st_shared_v4(dst + ((((uint32_t)(2 * i + 1)) ^ swz) << 4), hi);
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->full[rg.idx]));
                rg.next();
            }
        }
        // let every filter copy this thread issued land before the CTA exits
        if (threadIdx.x == 0 && *abort_flag) drain_ring(ctl->full, ST, b_issued, DRAIN_LIMIT_NS, a.status);
    } else if (warp < FIRST_EPI_WARP) {
        // ------------------------------------------------------------ MMA issuer
        ptx::setmaxnreg_dec<kTmemA ? TMEM_ISSUE_REGS : PRODUCER_REGS>();
        if (warp == MMA_WARP && lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_f16_f32(MT, NT);
            // stage s descriptors = stage 0 descriptors + s * (stage bytes >> 4)
            const uint64_t adesc0 = ptx::smem_desc_sw128(a_smem);
            const uint64_t bdesc0 = ptx::smem_desc_sw128(b_smem);
            Ring<ST> rg;
            uint32_t gi = 0;
            bool ok = true;
            if (kResB) ok = wait_phase(ptx::smem_addr(&ctl->b_res), 0, abort_flag, limit, a.status);
            for (int u = bid; u < a.num_units && ok; u += gdim) {
                const Unit w = unit_at(u, a.full_units, a.splits, a.k_steps);
                const int kn = w.ke - w.kb;
                const int ng = groups_of(kn);
                for (int g = 0; g < ng && ok; ++g) {
                    const int js = (int)(((int64_t)g * kn) / ng);
                    const int je = (int)(((int64_t)(g + 1) * kn) / ng);
                    const uint32_t slot = gi % NSLOT;
                    const uint32_t aph = (gi / NSLOT) & 1u;
                    if (!wait_phase(ptx::smem_addr(&ctl->acc_empty[slot]), aph ^ 1u, abort_flag, limit, a.status)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + slot * NT;
                    for (int j = js; j < je; ++j) {
                        // the stage's operands were published by TMA (complete_tx) or
                        // by producer stores followed by fence.proxy.async and the
                        // barrier arrive; waiting on the barrier orders them before
                        // the MMAs (no tcgen05 fence: nothing tcgen05-side to order)
                        if (!wait_phase(ptx::smem_addr(&ctl->full[rg.idx]), rg.phase, abort_flag, limit, a.status)) {
                            ok = false;
                            break;
                        }
                        const uint64_t adesc = adesc0 + (uint64_t)(rg.idx * (A_BYTES >> 4));
                        // kTmemA: the converters' tensor-memory stores are
                        // ordered before the MMAs by their fence, the barrier
                        // and this fence
                        if (kTmemA) ptx::tc_fence_after();
                        // resident filter: the block of this k-step
                        const uint64_t bdesc = kResB ? bdesc0 + (uint64_t)((w.kb + j) * (B_BYTES >> 4))
                                                     : bdesc0 + (uint64_t)(rg.idx * (B_BYTES >> 4));
#pragma unroll
                        for (int kk = 0; kk < KS / 16; ++kk) {
                            // advance 16 f16 = 32 bytes along K inside the swizzled row
                            // (8 columns in tensor memory)
                            if (kTmemA)
                                ptx::mma_f16_ts(d_tmem, tmem_base + (uint32_t)(Cfg::TMEM_A_COL + rg.idx * 32 + 8 * kk),
                                                bdesc + (uint64_t)(2 * kk), idesc, (j > js || kk > 0) ? 1u : 0u);
                            else
                                ptx::mma_f16_ss(d_tmem, adesc + (uint64_t)(2 * kk), bdesc + (uint64_t)(2 * kk), idesc,
                                                (j > js || kk > 0) ? 1u : 0u);
                        }
                        ptx::mma_commit(ptx::smem_addr(&ctl->empty[rg.idx]));
                        rg.next();
                    }
                    if (!ok) break;
                    ptx::mma_commit(ptx::smem_addr(&ctl->acc_full[slot]));
                    ++gi;
                }
            }
            // all MMAs issued by this thread complete before tensor memory is freed
            ptx::mma_commit(ptx::smem_addr(&ctl->mma_done));
            (void)drain_phase(ptx::smem_addr(&ctl->mma_done), 0, limit, a.status);
        } else if (kTma && (warp == A_ISSUER_WARP || (Cfg::A_ISSUERS == 2 && warp == A_ISSUER_WARP2)) && lane == 0) {
            const int issuer = warp == A_ISSUER_WARP ? 0 : 1;
            // im2col tiles: 128 consecutive output pixels x 64 channels of one
            // tap; the map's bounding box turns pixel order into window
            // origins (stride and pre-padding), the tap enters as the pixel
            // offset (r*dil_h, s*dil_w), and out-of-image reads are zeros
            Ring<STG> rs;
            int64_t issued = 0;
            bool ok = true;
            const int pq = a.P * a.Q;
            for (int u = bid; u < a.num_units && ok; u += gdim) {
                const Unit wu = unit_at(u, a.full_units, a.splits, a.k_steps);
                const int kn = wu.ke - wu.kb;
                const int m0 = fdiv(wu.tile, a.fd_nt) * MT;
                const int n0 = fdiv(m0, a.fd_pq);
                const int rem = m0 - n0 * pq;
                const int p0 = fdiv(rem, a.fd_q);
                const int q0 = rem - p0 * a.Q;
                const int w0 = q0 * a.str_w - a.pad_w;
                const int h0 = p0 * a.str_h - a.pad_h;
                // kNchw: the tile's pixels lie on output rows p0, p0 + 1, ...
                // (into the next image past P - 1), one image-row box each
                const int nrows = kNchw ? fdiv(q0 + MT - 1, a.fd_q) + 1 : 1;
                const uint32_t box_bytes = (uint32_t)(KS * a.W);
                // k-step kb + j, held as (tap row r, tap column s, channel
                // block cb) and advanced without divisions (the issuing
                // thread's loop is on every k-step's path)
                const int tap = fdiv(wu.kb, a.fd_cs);
                int cb = wu.kb - tap * a.c_steps;
                int r = fdiv(tap, a.fd_s);
                int s = tap - r * a.S;
#pragma unroll 1
                for (int j = 0; j < kn; ++j) {
                    // every issuer walks the sequence and issues into its own
                    // slots (never more than one phase ahead on a slot: issuers
                    // <= slots)
                    if (Cfg::A_ISSUERS == 1 || rs.idx % Cfg::A_ISSUERS == issuer) {
                        if (!wait_phase(ptx::smem_addr(&ctl->stg_empty[rs.idx]), rs.phase ^ 1u, abort_flag, limit,
                                        a.status, kIssuerBackoffNs)) {
                            ok = false;
                            break;
                        }
                        const uint32_t bar = ptx::smem_addr(&ctl->stg_full[rs.idx]);
                        if (kNchw) {
                            // whole image rows h = p*stride_h - pre_h + r*dil_h of
                            // channels cb*64.., boxes {W, 1, 64, 1} of the NCHW map
                            // (rows outside the image and images past N read as zeros)
                            ptx::mbar_arrive_expect_tx(bar, (uint32_t)nrows * box_bytes);
                            int pb = p0, nb = n0;
#pragma unroll 1
                            for (int b = 0; b < nrows; ++b) {
                                ptx::tma_load_4d(stg_smem + rs.idx * STG_SLOT + (uint32_t)b * box_bytes, &a.tmap_x, 0,
                                                 pb * a.str_h - a.pad_h + r * a.dil_h, cb * KS, nb, bar);
                                if (++pb == a.P) {
                                    pb = 0;
                                    ++nb;
                                }
                            }
                        } else if (a.a_rows) {
                            ptx::mbar_arrive_expect_tx(bar, STG_BYTES);
                            ptx::tma_load_2d(stg_smem + rs.idx * STG_SLOT, &a.tmap_x, cb * KS, m0, bar);
                        } else {
                            ptx::mbar_arrive_expect_tx(bar, STG_BYTES);
                            ptx::tma_load_im2col_4d(stg_smem + rs.idx * STG_SLOT, &a.tmap_x, cb * KS, w0, h0, n0,
                                                    (uint16_t)(s * a.dil_w), (uint16_t)(r * a.dil_h), bar);
                        }
                    }
                    ++issued;
                    rs.next();
                    if (++cb == a.c_steps) {
                        cb = 0;
                        if (++s == a.S) {
                            s = 0;
                            ++r;
                        }
                    }
                }
            }
            if (*abort_flag) drain_ring_owned(ctl->stg_full, STG, issued, issuer, Cfg::A_ISSUERS, limit, a.status);
        } else if (kResB && warp == B_ISSUER_WARP && lane == 0) {
            // every filter block of the call (one tile of output channels),
            // once, onto one barrier; then wait for them so that no copy is
            // in flight when the CTA ends
            const uint32_t bar = ptx::smem_addr(&ctl->b_res);
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)(a.k_steps * B_BYTES));
            for (int j = 0; j < a.k_steps; ++j)
                ptx::bulk_copy_g2s(b_smem + j * B_BYTES, a.wp + (size_t)j * B_BYTES, B_BYTES, bar);
            (void)drain_phase(bar, 0, limit, a.status);
        } else if (kSelfB && warp == B_ISSUER_WARP && lane == 0) {
            // int8 filter tiles by TMA, in the k-step order of the image
            // tiles: for tap (r, s) and channel block cb the box
            // {64 channels, 1, 1, NT rows} of the {C, S, R, K} map at
            // (cb*64, s, r, nt*NT), the taps flipped (S-1-s, R-1-r) for
            // CONVOLUTION; channels past C and rows past K read as zeros
            Ring<(Cfg::BSTG > 0 ? Cfg::BSTG : 1)> rb;
            int64_t issued = 0;
            bool ok = true;
            for (int u = bid; u < a.num_units && ok; u += gdim) {
                const Unit wu = unit_at(u, a.full_units, a.splits, a.k_steps);
                const int nt = wu.tile - fdiv(wu.tile, a.fd_nt) * a.n_tiles;
                for (int jr = wu.kb; jr < wu.ke; ++jr) {
                    const int tap = fdiv(jr, a.fd_cs);
                    const int cb = jr - tap * a.c_steps;
                    const int r = fdiv(tap, a.fd_s);
                    const int s = tap - r * a.S;
                    if (!wait_phase(ptx::smem_addr(&ctl->bstg_empty[rb.idx]), rb.phase ^ 1u, abort_flag, limit,
                                    a.status, kIssuerBackoffNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = ptx::smem_addr(&ctl->bstg_full[rb.idx]);
                    ptx::mbar_arrive_expect_tx(bar, (uint32_t)Cfg::BSTG_SLOT);
                    ptx::tma_load_4d(bstg_smem + rb.idx * Cfg::BSTG_SLOT, &a.tmap_w, cb * KS, a.mode ? a.S - 1 - s : s,
                                     a.mode ? a.R - 1 - r : r, nt * NT, bar);
                    ++issued;
                    rb.next();
                }
            }
            if (*abort_flag) drain_ring(ctl->bstg_full, Cfg::BSTG, issued, limit, a.status);
        } else if (kTma && warp == B_ISSUER_WARP && lane == 0) {
            // pre-swizzled f16 filter blocks, one bulk copy per k-step, in the
            // k-step order of the image tiles
            Ring<ST> rb;
            int64_t issued = 0;
            bool ok = true;
            for (int u = bid; u < a.num_units && ok; u += gdim) {
                const Unit wu = unit_at(u, a.full_units, a.splits, a.k_steps);
                const int nt = wu.tile - fdiv(wu.tile, a.fd_nt) * a.n_tiles;
                const uint8_t *blk = a.wp + (size_t)nt * a.k_steps * (size_t)B_BYTES;
                for (int jr = wu.kb; jr < wu.ke; ++jr) {
                    if (!wait_phase(ptx::smem_addr(&ctl->empty[rb.idx]), rb.phase ^ 1u, abort_flag, limit,
                                    a.status, kIssuerBackoffNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bar = ptx::smem_addr(&ctl->full[rb.idx]);
                    ptx::mbar_arrive_expect_tx(bar, B_BYTES);
                    ptx::bulk_copy_g2s(b_smem + rb.idx * B_BYTES, blk + (size_t)jr * B_BYTES, B_BYTES, bar);
                    ++issued;
                    rb.next();
                }
            }
            if (*abort_flag) drain_ring(ctl->full, ST, issued, DRAIN_LIMIT_NS, a.status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        ptx::setmaxnreg_inc<EPILOGUE_REGS>();
        const int quad = warp & 3;                      // tensor-memory lanes this warp may access
        const int col0 = ((warp - FIRST_EPI_WARP) >> 2) * HALF;  // this warp's half of the columns
        // the tile row (pixel) in this thread's tensor-memory lane: the lane
        // itself, or, for NCHW-row image stages, 4*(lane%8) + lane/8
        const int prow = kNchw ? (((lane & 7) << 2) | (lane >> 3)) : lane;
        const int row = quad * 32 + prow;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)col0;
        // output staging buffer of store ch: alternating between two (the
        // last tile of a one-buffer variant starts on the second, which no
        // store has read yet), or the one; and the wait for the store that
        // last read it
        auto epi_buf_index = [](int ch, bool two) -> uint32_t {
            return Cfg::EPI_BUFS == 2 ? (uint32_t)(ch & 1) : (two ? (uint32_t)((ch + 1) & 1) : 0u);
        };
        auto epi_wait_buffer = [](bool two) {
            if (two)
                ptx::bulk_wait_group_read<1>();
            else
                ptx::bulk_wait_group_read<0>();
        };
        uint32_t gi = 0;
        bool ok = true;
        for (int u = bid; u < a.num_units && ok; u += gdim) {
            const Unit wu = unit_at(u, a.full_units, a.splits, a.k_steps);
            const int ng = groups_of(wu.ke - wu.kb);
            const int mt = fdiv(wu.tile, a.fd_nt);
            const int nt = wu.tile - mt * a.n_tiles;
            const int m = mt * MT + row;
            const bool valid = m < a.m_total;
            int64_t yoff = 0;
            if (valid) {
                const int pq = a.P * a.Q;
                const int n = fdiv(m, a.fd_pq);
                const int rem = m - n * pq;
                const int p = fdiv(rem, a.fd_q);
                const int q = rem - p * a.Q;
                yoff = (int64_t)n * a.ys_n + (int64_t)p * a.ys_p + (int64_t)q * a.ys_q;
            }
            // bias[k] (int32) for this warp's HALF columns: each lane loads
            // HALF/32 of them, and the warp passes them round with shuffles
            // when it adds them.  Loaded before the accumulators are waited
            // for, so that the load's latency hides behind the tile's
            // main loop instead of lengthening the epilogue.
            int32_t bv[HALF / 32];
            if (a.bias && wu.split < 0) {
                const int kb = nt * NT + col0;
#pragma unroll
                for (int j = 0; j < HALF / 32; ++j) {
                    const int k = kb + j * 32 + lane;
                    bv[j] = k < a.K ? __ldg(a.bias + k) : 0;
                }
            }
            int32_t acc[HALF];
#pragma unroll
            for (int i = 0; i < HALF; ++i) acc[i] = 0;
            for (int g = 0; g < ng; ++g) {
                const uint32_t slot = gi % NSLOT;
                const uint32_t aph = (gi / NSLOT) & 1u;
                // tcgen05.ld is warp-collective: the whole warp proceeds or stops together
                const bool got =
                    wait_phase(ptx::smem_addr(&ctl->acc_full[slot]), aph, abort_flag, limit, a.status, kEpilogueBackoffNs);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // 32-column tensor-memory loads, LD_BATCH in flight per wait
                // (two where the registers allow: 64-column halves)
                constexpr int LD_BATCH = HALF <= 64 ? 2 : 1;
#pragma unroll
                for (int cc = 0; cc < HALF / 32; cc += LD_BATCH) {
                    uint32_t v[LD_BATCH][32];
#pragma unroll
                    for (int b = 0; b < LD_BATCH; ++b)
                        ptx::tmem_ld_32x32b_x32(lane_base + slot * NT + (cc + b) * 32, v[b]);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int b = 0; b < LD_BATCH; ++b)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            acc[(cc + b) * 32 + i] += __float2int_rn(__uint_as_float(v[b][i]));
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_addr(&ctl->acc_empty[slot]));
                ++gi;
            }
            if (!ok) break;
            const bool two_bufs = Cfg::EPI_BUFS == 2 || (Cfg::EPI_ALLOC == 2 && u + gdim >= a.num_units);
            if (wu.split >= 0) {
                // one run of a cut tile: its raw int32 sums go to the
                // workspace as int4 quads, [cut tile][split][column quad][row]
                // (a warp's store covers 32 consecutive rows: 512 contiguous
                // bytes); the reduction kernel adds the runs and finishes the
                // tile
                int4 *dst = reinterpret_cast<int4 *>(
                                a.tail_part + ((size_t)(wu.tile - a.full_units) * a.splits + wu.split) * MT * NT) +
                            (col0 / 4) * MT + row;
#pragma unroll
                for (int c4 = 0; c4 < HALF / 4; ++c4)
                    __stcg(dst + (size_t)c4 * MT,
                           make_int4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]));
                continue;
            }
            // epilogue arithmetic, once: + bias[k] (int32 wrap-around), then
            // ReLU.  All lanes of the warp hold the same HALF columns.
            if (a.bias) {
#pragma unroll
                for (int i = 0; i < HALF; ++i)
                    acc[i] = (int32_t)((uint32_t)acc[i] + (uint32_t)__shfl_sync(0xffffffffu, bv[i / 32], i % 32));
            }
            if (a.relu) {
#pragma unroll
                for (int i = 0; i < HALF; ++i) acc[i] = max(acc[i], 0);
            }
            if (a.y_tma == 2) {
                // Channel-major output: the warp's 32 rows are 32 consecutive
                // pixels of one image (P*Q is a multiple of 32).  It stages
                // EPI_COLS channels x 32 pixels at a time as rows of 128
                // bytes, the lane holding pixel i writing position i of each
                // row (no bank conflicts), and one lane stores them as a {32 pixels,
                // EPI_COLS channels, 1 image} box; the map clips channels past
                // K and images past N.
                const int k0 = nt * NT + col0;
                const int m0w = mt * MT + quad * 32;
                const int pq = a.P * a.Q;
                const int img = fdiv(m0w, a.fd_pq);
                const int pix = m0w - img * pq;
                const uint32_t ebase = epi_smem + (uint32_t)(warp - FIRST_EPI_WARP) * (uint32_t)(Cfg::EPI_ALLOC * Cfg::EPI_BUF_BYTES);
#pragma unroll
                for (int ch = 0; ch < HALF / Cfg::EPI_COLS; ++ch) {
                    const uint32_t buf = ebase + epi_buf_index(ch, two_bufs) * Cfg::EPI_BUF_BYTES;
                    if (lane == 0) epi_wait_buffer(two_bufs);
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_COLS; ++c)
                        ptx::st_shared_b32(buf + (uint32_t)c * 128u + (uint32_t)prow * 4u,
                                           (uint32_t)acc[ch * Cfg::EPI_COLS + c]);
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&a.tmap_y, pix, k0 + ch * Cfg::EPI_COLS, img, buf);
                        ptx::bulk_commit_group();
                    }
                }
            } else if (a.y_tma && a.out_int8) {
                // int8 output: as below, with 64 one-byte columns per 64-byte
                // staged row
                const int k0 = nt * NT + col0;
                const int m0w = mt * MT + quad * 32;
                const uint32_t ebase = epi_smem + (uint32_t)(warp - FIRST_EPI_WARP) * (uint32_t)(Cfg::EPI_ALLOC * Cfg::EPI_BUF_BYTES);
                const uint32_t sw = ((uint32_t)prow >> 1) & 3u;
#pragma unroll
                for (int ch = 0; ch < HALF / 64; ++ch) {
                    const uint32_t buf = ebase + epi_buf_index(ch, two_bufs) * Cfg::EPI_BUF_BYTES;
                    if (lane == 0) epi_wait_buffer(two_bufs);
                    __syncwarp();
                    const uint32_t rowaddr = buf + (uint32_t)prow * 64u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t wv[4];
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            wv[q4] = 0;
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int i = ch * 64 + c * 16 + q4 * 4 + e;
                                wv[q4] |= (uint32_t)(uint8_t)requant_i8(acc[i], a.out_shift) << (8 * e);
                            }
                        }
                        ptx::st_shared_v4(rowaddr + ((((uint32_t)c) ^ sw) << 4), make_uint4(wv[0], wv[1], wv[2], wv[3]));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&a.tmap_y, k0 + ch * 64, m0w, buf);
                        ptx::bulk_commit_group();
                    }
                }
            } else if (a.y_tma) {
                // Rows of the tile are consecutive pixels with contiguous
                // channels: each warp stages 32 rows x EPI_COLS columns at a
                // time in shared memory (rows of EPI_COLS * 4 bytes; 16-byte
                // chunk c of row r at c ^ ((r >> 1) & 3), the 64-byte
                // swizzle, or at c ^ (r & 7), the 128-byte swizzle) and one
                // lane writes them with a TMA store, which also clips rows
                // past the last pixel and columns past K.  With two buffers
                // per warp they alternate; with one, each store waits for
                // the last to have read it.
                constexpr int CHUNKS = Cfg::EPI_COLS / 4;  // 16-byte chunks per staged row
                const int k0 = nt * NT + col0;
                const int m0w = mt * MT + quad * 32;
                const uint32_t ebase = epi_smem + (uint32_t)(warp - FIRST_EPI_WARP) * (uint32_t)(Cfg::EPI_ALLOC * Cfg::EPI_BUF_BYTES);
                const uint32_t sw = CHUNKS == 8 ? ((uint32_t)prow & 7u) : (((uint32_t)prow >> 1) & 3u);
#pragma unroll
                for (int ch = 0; ch < HALF / Cfg::EPI_COLS; ++ch) {
                    const uint32_t buf = ebase + epi_buf_index(ch, two_bufs) * Cfg::EPI_BUF_BYTES;
                    if (lane == 0) epi_wait_buffer(two_bufs);
                    __syncwarp();
                    const int i0 = ch * Cfg::EPI_COLS;
                    const uint32_t rowaddr = buf + (uint32_t)prow * (uint32_t)(Cfg::EPI_COLS * 4);
#pragma unroll
                    for (int c = 0; c < CHUNKS; ++c)
                        ptx::st_shared_v4(rowaddr + ((((uint32_t)c) ^ sw) << 4),
                                          make_uint4((uint32_t)acc[i0 + c * 4], (uint32_t)acc[i0 + c * 4 + 1],
                                                     (uint32_t)acc[i0 + c * 4 + 2], (uint32_t)acc[i0 + c * 4 + 3]));
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&a.tmap_y, k0 + ch * Cfg::EPI_COLS, m0w, buf);
                        ptx::bulk_commit_group();
                    }
                }
            } else if (valid && a.out_int8) {
                const int k0 = nt * NT + col0;
                int8_t *yrow = static_cast<int8_t *>(a.y) + yoff;
#pragma unroll
                for (int i = 0; i < HALF; ++i) {
                    const int k = k0 + i;
                    if (k < a.K) yrow[(int64_t)k * a.ys_k] = requant_i8(acc[i], a.out_shift);
                }
            } else if (valid) {
                const int k0 = nt * NT + col0;
                int32_t *yrow = static_cast<int32_t *>(a.y) + yoff;
#pragma unroll
                for (int c4 = 0; c4 < HALF / 4; ++c4) {
                    const int k = k0 + c4 * 4;
                    const int32_t o[4] = {acc[c4 * 4], acc[c4 * 4 + 1], acc[c4 * 4 + 2], acc[c4 * 4 + 3]};
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
        // the output stores must finish reading shared memory before the CTA
        // exits (their writes complete with the grid)
        if (a.y_tma && lane == 0) ptx::bulk_wait_group_read<0>();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == MMA_WARP) ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

template <int NT, bool kTma, bool kResB, bool kTmemA, bool kNchw, bool kSelfB>
__global__ void __launch_bounds__(THREADS, 1) igemm_conv_kernel(const __grid_constant__ IgemmArgs a) {
    conv_cta<NT, kTma, kResB, kTmemA, kNchw, kSelfB>(a, blockIdx.x, gridDim.x);
}

// Several convolutions of one kernel variant in one launch (the residue
// classes of a data gradient): CTAs cta_start[c] .. cta_start[c+1]-1 work
// on convolution c alone, each reading its own arguments.
constexpr int kMaxGroup = kIgemmMaxGroup;
struct IgemmGroup {
    IgemmArgs cls[kMaxGroup];
    int32_t cta_start[kMaxGroup + 1];
    int32_t n;
};

template <int NT, bool kTma, bool kResB, bool kTmemA, bool kNchw, bool kSelfB>
__global__ void __launch_bounds__(THREADS, 1) igemm_conv_group_kernel(const __grid_constant__ IgemmGroup g) {
    int c = 0;
    while (c + 1 < g.n && (int)blockIdx.x >= g.cta_start[c + 1]) ++c;
    conv_cta<NT, kTma, kResB, kTmemA, kNchw, kSelfB>(g.cls[c], (int)blockIdx.x - g.cta_start[c],
                                      g.cta_start[c + 1] - g.cta_start[c]);
}

// ---------------------------------------------------------------- filter repack
// Writes B blocks: for n-tile nt and k-step j, NT rows (output channels) of
// 64 f16 (channels cb*64.. of tap (r, s) = divmod(j / c_steps, S), flipped for
// CONVOLUTION), each row's 16-byte chunk i stored at chunk position
// i ^ (row % 8): the image of the shared-memory stage, copied as one block.
// One filter to repack: its view (base, element strides [K][C][R][S]), the
// convolution's sizes and mode, and the plan's block geometry.
// kperm: the K order of the NCHW-row variants, which within every 16
// channels puts channel 4a + b at position 4b + a.
struct PackFilterJob {
    const int8_t *w;
    int64_t ws0, ws1, ws2, ws3;
    int32_t K, C, R, S, mode, c_steps, k_steps, n_tiles, nt_rows, kperm;
    FastDiv fd_rows, fd_ksteps, fd_csteps, fd_s;  // by nt_rows, k_steps, c_steps, S
    uint8_t *wp;
};

__device__ __forceinline__ int64_t pack_filter_items(const PackFilterJob &j) {
    return (int64_t)j.n_tiles * j.k_steps * j.nt_rows * 8;
}

// Item idx of a repack: 16-byte chunk (idx & 7) of block row idx >> 3.
// kWide: a repack of 2^31 items or more (64-bit index arithmetic); otherwise
// the row, k-step, tap and channel block come from multiply-high divisions.
template <bool kWide>
__device__ __forceinline__ void pack_filter_item(const PackFilterJob &jb, int64_t idx) {
    const int nt_rows = jb.nt_rows, k_steps = jb.k_steps, c_steps = jb.c_steps;
    const int chunk = (int)(idx & 7);
    int64_t t2;
    int nl, j, nt, tap, r;
    if (kWide) {
        const int64_t t = idx >> 3;
        nl = (int)(t % nt_rows);
        t2 = t / nt_rows;
        j = (int)(t2 % k_steps);
        nt = (int)(t2 / k_steps);
        tap = j / c_steps;
        r = tap / jb.S;
    } else {
        const int t = (int)(idx >> 3);
        const int q = fdiv(t, jb.fd_rows);
        nl = t - q * nt_rows;
        t2 = q;
        nt = fdiv(q, jb.fd_ksteps);
        j = q - nt * k_steps;
        tap = fdiv(j, jb.fd_csteps);
        r = fdiv(tap, jb.fd_s);
    }
    const int k = nt * nt_rows + nl;
    const int cb = j - tap * c_steps;
    const int s = tap - r * jb.S;
    const int rf = jb.mode ? jb.R - 1 - r : r;
    const int sf = jb.mode ? jb.S - 1 - s : s;
    const int c0 = cb * KS + chunk * 8;
    const int8_t *w = jb.w;
    uint32_t words[4];
    const int64_t off = (int64_t)k * jb.ws0 + (int64_t)c0 * jb.ws1 + (int64_t)rf * jb.ws2 + (int64_t)sf * jb.ws3;
    if (!jb.kperm && k < jb.K && c0 + 8 <= jb.C && jb.ws1 == 1 && ((uintptr_t)(w + off) & 7) == 0) {
        // eight channels contiguous in memory: one 8-byte load
        const uint2 v = *reinterpret_cast<const uint2 *>(w + off);
        const uint32_t lo = v.x ^ 0x80808080u, hi = v.y ^ 0x80808080u;
        words[0] = cvt_pair(lo, 0x4140);
        words[1] = cvt_pair(lo, 0x4342);
        words[2] = cvt_pair(hi, 0x4140);
        words[3] = cvt_pair(hi, 0x4342);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            unsigned short hv[2];
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const int kpos = chunk * 8 + 2 * e + b;  // position in the block's 64
                const int c = jb.kperm ? cb * KS + ((kpos & ~15) | ((kpos & 3) << 2) | ((kpos >> 2) & 3)) : c0 + 2 * e + b;
                int v = 0;
                if (k < jb.K && c < jb.C)
                    v = w[(int64_t)k * jb.ws0 + (int64_t)c * jb.ws1 + (int64_t)rf * jb.ws2 + (int64_t)sf * jb.ws3];
                hv[b] = __half_as_ushort(__int2half_rn(v));
            }
            words[e] = (uint32_t)hv[0] | ((uint32_t)hv[1] << 16);
        }
    }
    uint8_t *dst = jb.wp + ((t2 * nt_rows + nl) * 128) + (((chunk ^ (nl & 7))) << 4);
    *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
}

template <bool kWide>
__global__ void igemm_pack_filter_kernel(const __grid_constant__ PackFilterJob jb) {
    ptx::launch_dependents();
    const int64_t total = pack_filter_items(jb);
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x)
        pack_filter_item<kWide>(jb, idx);
}

// Shared tiles of the transposing copies below: 64 rows of 64 bytes, 4 bytes
// of padding per row.
constexpr int kBmPitch = 68;

// The same repack for a filter whose output channels are adjacent bytes (K
// stride 1: the weight gradient's loss gradient as its filter, a data
// gradient's exchanged filter): a block takes 64 rows (output channels) x
// the 64 channels of one k-step, by 16-byte loads of 64 consecutive rows per
// channel (four threads per channel), a transpose through shared memory,
// and 16-byte stores of 8 f16 channels per row into the pre-swizzled block.
// Needs 16-byte aligned channel, tap-row and tap strides and base; rows past
// K and channels past C are zeros.
__global__ void __launch_bounds__(256) igemm_pack_filter_k_minor_kernel(const __grid_constant__ PackFilterJob jb) {
    ptx::launch_dependents();
    __shared__ __align__(16) uint8_t tile[64 * kBmPitch];
    const int t = threadIdx.x;
    const int row_blocks = jb.nt_rows / 64;
    const int64_t total = (int64_t)jb.n_tiles * jb.k_steps * row_blocks;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int rb = (int)(b % row_blocks);
        const int64_t t2 = b / row_blocks;  // block index nt * k_steps + j
        const int nt = (int)(t2 / jb.k_steps);
        const int j = (int)(t2 - (int64_t)nt * jb.k_steps);
        const int tap = j / jb.c_steps;
        const int cb = j - tap * jb.c_steps;
        const int r = tap / jb.S, s = tap - (tap / jb.S) * jb.S;
        const int rf = jb.mode ? jb.R - 1 - r : r;
        const int sf = jb.mode ? jb.S - 1 - s : s;
        const int k0 = nt * jb.nt_rows + rb * 64;
        {
            const int cl = t >> 2, q = t & 3;
            const int c = cb * KS + cl;
            const int k = k0 + 16 * q;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (c < jb.C) {
                const int8_t *src = jb.w + (int64_t)c * jb.ws1 + (int64_t)rf * jb.ws2 + (int64_t)sf * jb.ws3 + k;
                if (k + 16 <= jb.K) {
                    v = __ldg(reinterpret_cast<const uint4 *>(src));
                } else {
                    uint32_t wd[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (k + e < jb.K) wd[e >> 2] |= (uint32_t)(uint8_t)src[e] << (8 * (e & 3));
                    v = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
            }
            uint32_t *row = reinterpret_cast<uint32_t *>(tile + cl * kBmPitch + 16 * q);
            row[0] = v.x; row[1] = v.y; row[2] = v.z; row[3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int item = t + 256 * i;
            const int nl = rb * 64 + (item >> 3), chunk = item & 7;
            uint32_t words[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c0 = chunk * 8 + 2 * e;
                const int v0 = (int8_t)tile[c0 * kBmPitch + (item >> 3)];
                const int v1 = (int8_t)tile[(c0 + 1) * kBmPitch + (item >> 3)];
                words[e] = (uint32_t)__half_as_ushort(__int2half_rn(v0)) |
                           ((uint32_t)__half_as_ushort(__int2half_rn(v1)) << 16);
            }
            uint8_t *dst = jb.wp + ((t2 * jb.nt_rows + nl) * 128) + ((chunk ^ (nl & 7)) << 4);
            *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        }
        __syncthreads();
    }
}

// The weight gradient folded over T output columns (see WgradFold): the
// image copy X'' and the folded loss-gradient repack, each a transpose
// through a shared tile of 64 x 64 bytes like the two kernels above.
struct WgradFoldArgs {
    const int8_t *x;
    int64_t xs0, xs1, xs2, xs3;
    const int8_t *dy;
    int64_t ys0, ys1, ys2, ys3;
    int64_t N, C, H, W, K, P, Q, T, Q2, U, c16, pre_w, stride_w;
    int32_t x_vec, dy_vec;  // 16-byte loads allowed (unit stride along the loaded run, aligned)
    int32_t nt_rows, n_tiles, k_steps;
    int8_t *x2;
    uint8_t *wp;
};

// Block (image block cb of 64 images c, row h, column u): tile[ch][c] holds
// X''[c][h][u][ch] for the block's images.
__global__ void __launch_bounds__(256) igemm_wgrad_fold_image_kernel(const __grid_constant__ WgradFoldArgs f) {
    ptx::launch_dependents();
    __shared__ __align__(16) uint8_t tile[64 * kBmPitch];
    const int t = threadIdx.x;
    const int64_t cblocks = (f.C + 63) / 64;
    const int64_t total = cblocks * f.H * f.U;
    const int64_t tn = f.T * f.N;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int64_t u = b % f.U;
        const int64_t t2 = b / f.U;
        const int64_t h = t2 % f.H;
        const int64_t c0 = (t2 / f.H) * 64;
        {
            const int ch = t >> 2, q = t & 3;
            const int64_t c = c0 + 16 * q;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (ch < tn && ch < f.c16) {
                const int64_t n = ch % f.N, tt = ch / f.N;
                const int64_t w = u - f.pre_w + tt * f.stride_w;
                if (w >= 0 && w < f.W && c < f.C) {
                    const int8_t *src = f.x + n * f.xs0 + c * f.xs1 + h * f.xs2 + w * f.xs3;
                    if (f.x_vec && c + 16 <= f.C) {
                        v = __ldg(reinterpret_cast<const uint4 *>(src));
                    } else {
                        uint32_t wd[4] = {0, 0, 0, 0};
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c + e < f.C) wd[e >> 2] |= (uint32_t)(uint8_t)src[e * f.xs1] << (8 * (e & 3));
                        v = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    }
                }
            }
            uint32_t *row = reinterpret_cast<uint32_t *>(tile + ch * kBmPitch + 16 * q);
            row[0] = v.x; row[1] = v.y; row[2] = v.z; row[3] = v.w;
        }
        __syncthreads();
        {
            const int cl = t >> 2, cq = t & 3;
            const int64_t c = c0 + cl;
            if (c < f.C && 16 * cq < f.c16) {
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t word = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) word |= (uint32_t)tile[(16 * cq + 4 * e + k) * kBmPitch + cl] << (8 * k);
                    wd[e] = word;
                }
                *reinterpret_cast<uint4 *>(f.x2 + ((c * f.H + h) * f.U + u) * f.c16 + 16 * cq) =
                    make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
        }
        __syncthreads();
    }
}

// Block (n-tile nt, k-step j = tap (p, q2), row block rb of 64 output
// channels k): tile[ch][k] holds the folded loss gradient's channel ch, and
// the block's 64 pre-swizzled f16 rows are written from it.
__global__ void __launch_bounds__(256) igemm_wgrad_fold_filter_kernel(const __grid_constant__ WgradFoldArgs f) {
    ptx::launch_dependents();
    __shared__ __align__(16) uint8_t tile[64 * kBmPitch];
    const int t = threadIdx.x;
    const int row_blocks = f.nt_rows / 64;
    const int64_t total = (int64_t)f.n_tiles * f.k_steps * row_blocks;
    const int64_t tn = f.T * f.N;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int rb = (int)(b % row_blocks);
        const int64_t t2 = b / row_blocks;  // block index nt * k_steps + j
        const int64_t nt = t2 / f.k_steps;
        const int64_t j = t2 - nt * f.k_steps;
        const int64_t p = j / f.Q2, q2 = j - (j / f.Q2) * f.Q2;
        const int64_t k0 = nt * f.nt_rows + rb * 64;
        {
            const int ch = t >> 2, q = t & 3;
            const int64_t k = k0 + 16 * q;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (ch < tn && ch < f.c16) {
                const int64_t n = ch % f.N, qq = f.T * q2 + ch / f.N;
                if (qq < f.Q && k < f.K) {
                    const int8_t *src = f.dy + n * f.ys0 + k * f.ys1 + p * f.ys2 + qq * f.ys3;
                    if (f.dy_vec && k + 16 <= f.K) {
                        v = __ldg(reinterpret_cast<const uint4 *>(src));
                    } else {
                        uint32_t wd[4] = {0, 0, 0, 0};
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (k + e < f.K) wd[e >> 2] |= (uint32_t)(uint8_t)src[e * f.ys1] << (8 * (e & 3));
                        v = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    }
                }
            }
            uint32_t *row = reinterpret_cast<uint32_t *>(tile + ch * kBmPitch + 16 * q);
            row[0] = v.x; row[1] = v.y; row[2] = v.z; row[3] = v.w;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int item = t + 256 * i;
            const int64_t nl = rb * 64 + (item >> 3);
            const int chunk = item & 7;
            uint32_t words[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c0 = chunk * 8 + 2 * e;
                const int v0 = (int8_t)tile[c0 * kBmPitch + (item >> 3)];
                const int v1 = (int8_t)tile[(c0 + 1) * kBmPitch + (item >> 3)];
                words[e] = (uint32_t)__half_as_ushort(__int2half_rn(v0)) |
                           ((uint32_t)__half_as_ushort(__int2half_rn(v1)) << 16);
            }
            uint8_t *dst = f.wp + ((t2 * f.nt_rows + nl) * 128) + ((chunk ^ (int)(nl & 7)) << 4);
            *reinterpret_cast<uint4 *>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        }
        __syncthreads();
    }
}

// Several repacks in one launch (the residue classes of a data gradient):
// the items of job i are end[i-1] .. end[i]-1 of the grid walk.
struct PackFilterJobs {
    PackFilterJob job[kMaxPackJobs];
    int64_t end[kMaxPackJobs];
    int32_t n;
};

template <bool kWide>
__global__ void igemm_pack_filter_group_kernel(const __grid_constant__ PackFilterJobs js) {
    ptx::launch_dependents();
    const int64_t total = js.end[js.n - 1];
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int i = 0;
        while (idx >= js.end[i]) ++i;
        pack_filter_item<kWide>(js.job[i], idx - (i ? js.end[i - 1] : 0));
    }
}

// ---------------------------------------------------------------- cut tiles
// Adds the runs of every cut tile (tiles tile0.. of the grid walk; raw int32
// sums in the workspace as int4 quads, [cut tile][split][column quad][row]),
// then applies bias, ReLU and the int8 requantisation like the main epilogue
// and stores the tile.  A block (256 threads) takes 32 rows x 32 columns of
// one cut tile, one quad per thread: each warp reads 32 consecutive rows of
// one quad (512 contiguous bytes per run), four runs' loads in flight; the
// sums go through a shared tile so that the stores run with columns fastest
// when the output's channels are contiguous (a thread stores four channels
// of one pixel, eight threads a pixel's 32), rows fastest otherwise
// (consecutive pixels of one channel).
constexpr int kRedRows = 32, kRedCols = 32, kRedPitch = kRedCols + 4;  // int32 per shared row
__global__ void __launch_bounds__(256) igemm_split_reduce_kernel(const int32_t *part, int32_t tile0,
                                                                 int32_t tiles, int32_t splits,
                                                                 int32_t n_tiles, int32_t nt_cols, int32_t m_total,
                                                                 int32_t K, int32_t P, int32_t Q, int64_t ys_n,
                                                                 int64_t ys_k, int64_t ys_p, int64_t ys_q, void *y,
                                                                 int32_t out_int8, int32_t out_shift,
                                                                 const int32_t *bias, int32_t relu) {
    __shared__ __align__(16) int32_t sums[kRedRows * kRedPitch];
    // launched as a programmatic dependent of the convolution: nothing is
    // read before its writes are visible
    ptx::grid_dependency_wait();
    const int qblocks = nt_cols / kRedCols, rblocks = MT / kRedRows;
    const int64_t total = (int64_t)tiles * qblocks * rblocks;
    const bool chan_fast = ys_k == 1;
    const int pq = P * Q;
    const size_t run_quads = (size_t)MT * nt_cols / 4;
    const int lr = threadIdx.x % kRedRows, lq = threadIdx.x / kRedRows;  // this thread's row and quad
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int rb = (int)(b % rblocks);
        const int64_t t = b / rblocks;
        const int qb = (int)(t % qblocks);
        const int ct = (int)(t / qblocks);  // cut tile
        const int tile = tile0 + ct;
        const int mt = tile / n_tiles;
        const int nt = tile - mt * n_tiles;
        const int4 *src = reinterpret_cast<const int4 *>(part + (size_t)ct * splits * MT * nt_cols) +
                          (size_t)(qb * (kRedCols / 4) + lq) * MT + rb * kRedRows + lr;
        int4 v = make_int4(0, 0, 0, 0);
#pragma unroll 4
        for (int sp = 0; sp < splits; ++sp) {
            const int4 x = __ldcg(src + sp * run_quads);
            v.x += x.x;
            v.y += x.y;
            v.z += x.z;
            v.w += x.w;
        }
        *reinterpret_cast<int4 *>(sums + lr * kRedPitch + lq * 4) = v;
        __syncthreads();
        if (chan_fast) {
            // thread = (row, 4 columns): one pixel decomposition, four
            // consecutive channels (16 bytes of int32 when aligned)
            const int row = threadIdx.x / (kRedCols / 4), c0 = (threadIdx.x % (kRedCols / 4)) * 4;
            const int m = mt * MT + rb * kRedRows + row;
            const int k0 = nt * nt_cols + qb * kRedCols + c0;
            if (m < m_total && k0 < K) {
                const int n = m / pq;
                const int rem = m - n * pq;
                const int p = rem / Q;
                const int q = rem - p * Q;
                const int64_t yoff = (int64_t)n * ys_n + (int64_t)p * ys_p + (int64_t)q * ys_q;
                int32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int32_t val = sums[row * kRedPitch + c0 + e];
                    if (bias && k0 + e < K) val = (int32_t)((uint32_t)val + (uint32_t)__ldg(bias + k0 + e));
                    o[e] = relu ? max(val, 0) : val;
                }
                if (!out_int8 && k0 + 3 < K && ((uintptr_t)(static_cast<int32_t *>(y) + yoff + k0) & 15) == 0) {
                    *reinterpret_cast<int4 *>(static_cast<int32_t *>(y) + yoff + k0) = make_int4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (k0 + e >= K) break;
                        if (out_int8)
                            static_cast<int8_t *>(y)[yoff + k0 + e] = requant_i8(o[e], out_shift);
                        else
                            static_cast<int32_t *>(y)[yoff + k0 + e] = o[e];
                    }
                }
            }
        } else {
            for (int i = threadIdx.x; i < kRedRows * kRedCols; i += blockDim.x) {
                const int row = i % kRedRows, col = i / kRedRows;  // consecutive pixels of one channel
                const int m = mt * MT + rb * kRedRows + row;
                const int k = nt * nt_cols + qb * kRedCols + col;
                if (m >= m_total || k >= K) continue;
                int32_t val = sums[row * kRedPitch + col];
                if (bias) val = (int32_t)((uint32_t)val + (uint32_t)__ldg(bias + k));
                if (relu) val = max(val, 0);
                const int n = m / pq;
                const int rem = m - n * pq;
                const int p = rem / Q;
                const int q = rem - p * Q;
                const int64_t off = (int64_t)n * ys_n + (int64_t)p * ys_p + (int64_t)q * ys_q + (int64_t)k * ys_k;
                if (out_int8)
                    static_cast<int8_t *>(y)[off] = requant_i8(val, out_shift);
                else
                    static_cast<int32_t *>(y)[off] = val;
            }
        }
        __syncthreads();  // the next block's sums overwrite the tile
    }
}

// ---------------------------------------------------------------- image repack
// Channels-last copy of an image with arbitrary strides: xp[((n*H+h)*W+w)*c16 + c]
// = x[n, c, row0 + row_step*h, w] for the H copied rows, channels C..c16-1
// zero.  One thread writes 16 channels of one pixel; threads of a warp take
// neighbouring pixels so that reads along W coalesce for NCHW.
__global__ void igemm_pack_image_kernel(const int8_t *x, int64_t xs0, int64_t xs1, int64_t xs2, int64_t xs3,
                                        int64_t N, int32_t C, int32_t H, int32_t W, int32_t row0, int32_t row_step,
                                        int32_t c16, int8_t *xp) {
    ptx::launch_dependents();
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
        const int8_t *src = x + n * xs0 + (int64_t)(row0 + (int64_t)row_step * h) * xs2 + (int64_t)w * xs3;
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

// The same copy for an image whose images (the batch index) are adjacent
// bytes, stride 1: the weight gradient's image, a channels-last image with
// its batch and channels exchanged.  A block takes 64 images x 64 channels
// of one pixel: 16-byte loads of 64 consecutive images per channel (four
// threads per channel), a transpose through shared memory, and 16-byte
// stores of 16 channels per image (four threads per image's 64 channels).
// Needs 16-byte aligned channel and pixel strides and base; channels from C
// up to c16 are zero.

__global__ void __launch_bounds__(256) igemm_pack_image_batch_minor_kernel(
    const int8_t *x, int64_t xs1, int64_t xs2, int64_t xs3, int64_t N, int32_t C, int32_t H, int32_t W,
    int32_t row0, int32_t row_step, int32_t c16, int8_t *xp) {
    ptx::launch_dependents();
    __shared__ __align__(16) uint8_t tile[64 * kBmPitch];
    const int t = threadIdx.x;
    const int64_t nblocks = (N + 63) / 64;
    const int cblocks = (c16 + 63) / 64;
    const int64_t pixels = (int64_t)H * W;
    const int64_t total = nblocks * pixels * cblocks;
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int cb = (int)(b % cblocks);
        const int64_t pb = b / cblocks;
        const int64_t pix = pb % pixels;
        const int64_t n0 = (pb / pixels) * 64;
        const int h = (int)(pix / W), w = (int)(pix - (int64_t)(pix / W) * W);
        // load: channel cl = t / 4, images n0 + 16q .. +15
        {
            const int cl = t >> 2, q = t & 3;
            const int c = cb * 64 + cl;
            const int64_t n = n0 + 16 * q;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (c < C) {
                const int8_t *src = x + (int64_t)c * xs1 + (int64_t)(row0 + (int64_t)row_step * h) * xs2 +
                                    (int64_t)w * xs3 + n;
                if (n + 16 <= N) {
                    v = __ldg(reinterpret_cast<const uint4 *>(src));
                } else {
                    uint32_t wd[4] = {0, 0, 0, 0};
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (n + e < N) wd[e >> 2] |= (uint32_t)(uint8_t)src[e] << (8 * (e & 3));
                    v = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                }
            }
            uint32_t *row = reinterpret_cast<uint32_t *>(tile + cl * kBmPitch + 16 * q);
            row[0] = v.x; row[1] = v.y; row[2] = v.z; row[3] = v.w;
        }
        __syncthreads();
        // store: image nl = t / 4, channels cb*64 + 16cq .. +15
        {
            const int nl = t >> 2, cq = t & 3;
            const int64_t n = n0 + nl;
            const int c0 = cb * 64 + 16 * cq;
            if (n < N && c0 < c16) {
                uint32_t wd[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint32_t word = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) word |= (uint32_t)tile[(16 * cq + 4 * e + k) * kBmPitch + nl] << (8 * k);
                    wd[e] = word;
                }
                *reinterpret_cast<uint4 *>(xp + (n * pixels + pix) * c16 + c0) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
            }
        }
        __syncthreads();
    }
}

// The same copy for images whose channels each hold their H x W pixels in one
// contiguous plane (NCHW-like, 16-byte aligned planes, H*W a multiple of 16):
// a transpose through shared memory.  A block takes 64 channels x 256 pixels
// of one image.  Loads: four threads per channel, 16-byte loads of 256
// contiguous pixels, stored as they are in a [channel][pixel] tile.  Stores:
// a thread takes 4 pixels x 16 channels, reads the 16 channels' 4-pixel words
// and transposes each 4 x 4 block of bytes with byte permutes, then writes
// each pixel's 16 channels; four neighbouring threads cover a pixel's 64
// channels (64 contiguous bytes of the channels-last copy).  Channels from C
// up to c16 are zero.
constexpr int kPackPix = 256, kPackCh = 64, kPackPitch = 272;  // pitch: 16-byte rows, 2-way conflicts at most on the tile stores

__device__ __forceinline__ void transpose4x4_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t (&o)[4]) {
    // o[i] = byte i of a, b, c, d
    const uint32_t ab_lo = __byte_perm(a, b, 0x5140), ab_hi = __byte_perm(a, b, 0x7362);
    const uint32_t cd_lo = __byte_perm(c, d, 0x5140), cd_hi = __byte_perm(c, d, 0x7362);
    o[0] = __byte_perm(ab_lo, cd_lo, 0x5410);
    o[1] = __byte_perm(ab_lo, cd_lo, 0x7632);
    o[2] = __byte_perm(ab_hi, cd_hi, 0x5410);
    o[3] = __byte_perm(ab_hi, cd_hi, 0x7632);
}

// HW: pixels per copied image (copied rows x W); copied row h is image row
// row0 + row_step*h (with row_step > 1, W is a multiple of 16 so that no
// 16-byte load crosses a row).
__global__ void __launch_bounds__(256) igemm_pack_image_planes_kernel(const int8_t *x, int64_t xs0, int64_t xs1,
                                                                      int64_t N, int32_t C, int32_t HW, int32_t W,
                                                                      int32_t row0, int32_t row_step, int32_t c16,
                                                                      int8_t *xp) {
    ptx::launch_dependents();
    __shared__ __align__(16) uint8_t tile[kPackCh * kPackPitch];
    const int ptiles = (HW + kPackPix - 1) / kPackPix;
    const int ctiles = (c16 + kPackCh - 1) / kPackCh;
    const int64_t total = N * ptiles * ctiles;
    const int cl = threadIdx.x >> 2, seg = threadIdx.x & 3;  // loads: channel row, 64-pixel segment
    const int cb = threadIdx.x & 3, q = threadIdx.x >> 2;    // stores: 16-channel block, 4-pixel quad
    for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
        const int ct = (int)(b % ctiles);
        const int64_t t = b / ctiles;
        const int pt = (int)(t % ptiles);
        const int64_t n = t / ptiles;
        const int p0 = pt * kPackPix, c0 = ct * kPackCh;
        const int c = c0 + cl;
        const int8_t *plane = x + n * xs0 + (int64_t)c * xs1;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int p = p0 + seg * 64 + j * 16;  // copied pixel: row p / W, column p % W
            int64_t off = p;
            if (row_step > 1) {
                const int h = p / W;
                off = (int64_t)(row0 + row_step * h) * W + (p - h * W);
            }
            v[j] = (c < C && p < HW) ? __ldg(reinterpret_cast<const uint4 *>(plane + off)) : make_uint4(0, 0, 0, 0);
        }
        __syncthreads();  // the previous tile's stores have read the buffer
#pragma unroll
        for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(tile + cl * kPackPitch + seg * 64 + j * 16) = v[j];
        __syncthreads();
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 16; ++k)
            w[k] = *reinterpret_cast<const uint32_t *>(tile + (cb * 16 + k) * kPackPitch + q * 4);
        uint32_t px[4][4];  // [pixel][channel word]
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            uint32_t o[4];
            transpose4x4_bytes(w[4 * m], w[4 * m + 1], w[4 * m + 2], w[4 * m + 3], o);
#pragma unroll
            for (int i = 0; i < 4; ++i) px[i][m] = o[i];
        }
        const int cc = c0 + cb * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = p0 + q * 4 + i;
            if (p < HW && cc < c16)
                *reinterpret_cast<uint4 *>(xp + (n * HW + p) * c16 + cc) =
                    make_uint4(px[i][0], px[i][1], px[i][2], px[i][3]);
        }
    }
}

inline int64_t align256(int64_t v) { return (v + 255) & ~255LL; }

constexpr int64_t kSplitMinKSteps = 64;  // only reductions at least this long are cut
constexpr int64_t kMinSplitSteps = 16;   // k-steps of the shortest run of a cut tile
constexpr int64_t kMaxSplits = 32;
constexpr int64_t kMinTailSteps = 4;     // k-steps of the shortest run of a last-round tile

template <int NT, bool kTma, bool kResB = false, bool kTmemA = false, bool kNchw = false, bool kSelfB = false>
conv_status launch_conv(const IgemmArgs &a, int grid, cudaStream_t st) {
    using Cfg = TileCfg<NT, kTma, kResB, kTmemA, kNchw, kSelfB>;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev].load()) {
        if (cudaFuncSetAttribute(igemm_conv_kernel<NT, kTma, kResB, kTmemA, kNchw, kSelfB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg::SMEM_BYTES) != cudaSuccess)
            return CONV_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true);
    }
    // a programmatic dependent of the previous kernel in the stream: its CTAs
    // may start (allocate, initialise barriers) while a repack kernel that
    // signals launch_dependents finishes, and wait for its writes in
    // grid_dependency_wait; behind any other kernel or copy it starts when
    // that completes, as without the attribute
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, igemm_conv_kernel<NT, kTma, kResB, kTmemA, kNchw, kSelfB>, a) != cudaSuccess) return CONV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

// The driver's im2col tensor-map encoder, looked up once through the runtime
// (no link against the driver library).
PFN_cuTensorMapEncodeIm2col_v12000 im2col_encoder() {
    static std::atomic<void *> fn{nullptr};
    static std::atomic<bool> tried{false};
    if (!tried.load()) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn.store(p);
        tried.store(true);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(fn.load());
}

// im2col map of a channels-last int8 image [N][H][W][C] (byte strides
// xs_n, xs_h, xs_w): each load brings 128 consecutive output pixels x 64
// channels (rows 64-byte swizzled with swizzle64, for the converters that
// write the image tile to tensor memory).  The bounding box runs from -pre to post - (taps-1)*dil along W
// and H so that its traversal at the convolution stride visits exactly the
// P x Q window origins.  Returns false when the map cannot express the call
// (stride above 8, corner or offset out of range, encoder unavailable).
// The geometry the kernel sees: the call's, or, for an image copy that
// keeps every row_step-th row from row0, the same convolution over the copy
// (h = row0 + row_step*h', so stride, dilation and pre-padding along H are
// divided by row_step: pre' = (pre + row0) / row_step, exact).
ConvGeom kernel_geom(const ConvGeom &g, const IgemmPlan &pl) {
    ConvGeom k = g;
    if (pl.pack_x && pl.row_step > 1) {
        k.H = pl.hp;
        k.str_h = g.str_h / pl.row_step;
        k.dil_h = g.R > 1 ? g.dil_h / pl.row_step : g.dil_h;
        k.pad_h = (g.pad_h + pl.row0) / pl.row_step;
    }
    return k;
}

// The limits of an im2col map that do not depend on the image's address:
// stride at most 8, bounding-box corners within [-128, 127], tap offsets
// within 16 bits.
bool im2col_geometry_ok(const ConvGeom &g) {
    if (g.str_h > 8 || g.str_w > 8) return false;
    const int64_t lo_w = -g.pad_w, lo_h = -g.pad_h;
    const int64_t hi_w = (g.Q - 1) * g.str_w + lo_w - (g.W - 1);  // = post_w - (S-1)*dil_w
    const int64_t hi_h = (g.P - 1) * g.str_h + lo_h - (g.H - 1);
    for (int64_t v : {lo_w, lo_h, hi_w, hi_h})
        if (v < -128 || v > 127) return false;
    return (g.R - 1) * g.dil_h <= 65535 && (g.S - 1) * g.dil_w <= 65535;
}

bool encode_im2col_map(const ConvGeom &g, const void *x, int64_t xs_n, int64_t xs_h, int64_t xs_w, int64_t c_dim,
                       bool swizzle64, CUtensorMap *map) {
    if (!im2col_geometry_ok(g)) return false;
    const int64_t lo_w = -g.pad_w, lo_h = -g.pad_h;
    const int64_t hi_w = (g.Q - 1) * g.str_w + lo_w - (g.W - 1);  // = post_w - (S-1)*dil_w
    const int64_t hi_h = (g.P - 1) * g.str_h + lo_h - (g.H - 1);
    if (((uintptr_t)x % 16) != 0 || xs_w % 16 || xs_h % 16 || xs_n % 16) return false;
    auto enc = im2col_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)c_dim, (cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.N};
    const cuuint64_t strides[3] = {(cuuint64_t)xs_w, (cuuint64_t)xs_h, (cuuint64_t)xs_n};
    const int lower[2] = {(int)lo_w, (int)lo_h};
    const int upper[2] = {(int)hi_w, (int)hi_h};
    const cuuint32_t estr[4] = {1, (cuuint32_t)g.str_w, (cuuint32_t)g.str_h, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(x), dims, strides, lower, upper,
                           (cuuint32_t)KS, (cuuint32_t)MT, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 tiled_encoder();

// 2-D map [pixels][channels] of a channels-last image whose pixels follow
// one another at xs_w bytes (dense rows): for a 1x1 filter with stride 1 and
// no padding, the image tile of output pixels m0.. is the box of rows m0..
// (128 rows x 64 channels: the same staging layout as the im2col load,
// 64-byte swizzled or not).
bool encode_rows_map(const ConvGeom &g, const void *x, int64_t xs_w, int64_t c_dim, bool swizzle64,
                     CUtensorMap *map) {
    const int64_t rows = g.N * g.H * g.W;
    if (((uintptr_t)x % 16) != 0 || xs_w % 16 || rows >= ((int64_t)1 << 32)) return false;
    auto enc = tiled_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)c_dim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)xs_w};
    const cuuint32_t box[2] = {(cuuint32_t)KS, (cuuint32_t)MT};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 4-D map {W, H, C, N} of an int8 image whose channels hold contiguous rows
// (byte strides xs[2], xs[1], xs[0]): box {W, 1, 64, 1}, one image row of
// 64 channels, no swizzle (the NCHW-row variants).
bool encode_nchw_rows_map(const ConvGeom &g, const void *x, CUtensorMap *map) {
    auto enc = tiled_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)g.W, (cuuint64_t)g.H, (cuuint64_t)g.C, (cuuint64_t)g.N};
    const cuuint64_t strides[3] = {(cuuint64_t)g.xs[2], (cuuint64_t)g.xs[1], (cuuint64_t)g.xs[0]};
    const cuuint32_t box[4] = {(cuuint32_t)g.W, 1, (cuuint32_t)KS, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(x), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 tiled_encoder() {
    static std::atomic<void *> fn{nullptr};
    static std::atomic<bool> tried{false};
    if (!tried.load()) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn.store(p);
        tried.store(true);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn.load());
}

// 2-D map [N*P*Q pixels][K channels] of the output when its pixels follow one
// another at a fixed stride with channels contiguous (NHWC, possibly with
// padded pixel rows): box 32 pixels x 64 bytes of channels (16 int32 or 64
// int8) with the 64-byte swizzle, or (wide, int32) 32 pixels x 32 int32 with
// the 128-byte swizzle.  Returns false for any other layout.
bool encode_output_map(const ConvGeom &g, const void *y, bool wide, CUtensorMap *map) {
    const int64_t esz = g.out_int8 ? 1 : 4;
    if (g.ys[1] != 1 && g.K > 1) return false;
    int64_t ps;  // element stride between consecutive pixels
    if (g.Q > 1) {
        ps = g.ys[3];
        if (g.P > 1 && g.ys[2] != g.Q * ps) return false;
        if (g.N > 1 && g.ys[0] != g.P * g.Q * ps) return false;
    } else if (g.P > 1) {
        ps = g.ys[2];
        if (g.N > 1 && g.ys[0] != g.P * ps) return false;
    } else {
        ps = g.N > 1 ? g.ys[0] : g.K;
    }
    const int64_t m_total = g.N * g.P * g.Q;
    if (ps < g.K || (ps * esz) % 16 != 0 || ((uintptr_t)y % 16) != 0) return false;
    if (m_total > ((int64_t)1 << 32) || (m_total > 1 && ps * esz >= ((int64_t)1 << 40))) return false;
    auto enc = tiled_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)g.K, (cuuint64_t)m_total};
    const cuuint64_t strides[1] = {(cuuint64_t)(ps * esz)};
    const bool w32 = wide && !g.out_int8;
    const cuuint32_t box[2] = {(cuuint32_t)(g.out_int8 ? 64 : (w32 ? 32 : 16)), 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, g.out_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_INT32, 2,
                           const_cast<void *>(y), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           w32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D map [N][K][P*Q] of an int32 output whose channels each hold their P*Q
// pixels contiguously (NCHW, possibly with padded channel or image strides):
// box 32 pixels x 16 (or, wide, 32) channels x 1 image, no swizzle.  Requires P*Q to be a
// multiple of 32, so that the 32 pixels of an epilogue warp never straddle
// two images and start 128 bytes aligned.  Returns false for any other
// layout.
bool encode_output_map_nchw(const ConvGeom &g, const void *y, bool wide, CUtensorMap *map) {
    if (g.out_int8) return false;
    const int64_t pq = g.P * g.Q;
    if (pq % 32 != 0) return false;
    if (g.Q > 1 && g.ys[3] != 1) return false;
    if (g.P > 1 && g.ys[2] != g.Q) return false;
    const int64_t ks = g.K > 1 ? g.ys[1] : pq;
    const int64_t ns = g.N > 1 ? g.ys[0] : ks * g.K;
    if (ks < pq || ns < ks * g.K || (ks * 4) % 16 != 0 || (ns * 4) % 16 != 0 || ((uintptr_t)y % 16) != 0) return false;
    if (pq >= ((int64_t)1 << 32) || ns * 4 >= ((int64_t)1 << 40)) return false;
    auto enc = tiled_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)pq, (cuuint64_t)g.K, (cuuint64_t)g.N};
    const cuuint64_t strides[2] = {(cuuint64_t)(ks * 4), (cuuint64_t)(ns * 4)};
    const cuuint32_t box[3] = {32, (cuuint32_t)(wide ? 32 : 16), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_INT32, 3, const_cast<void *>(y), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool igemm_supported(const ConvGeom &g) {
    const int64_t lim = (int64_t)1 << 30;
    if (g.H >= lim || g.W >= lim || g.P >= lim || g.Q >= lim) return false;
    if (g.pad_h >= (1 << 20) || g.pad_w >= (1 << 20) || g.pad_h <= -(1 << 20) || g.pad_w <= -(1 << 20) ||
        g.str_h >= (1 << 20) || g.str_w >= (1 << 20) || g.dil_h >= (1 << 20) || g.dil_w >= (1 << 20))
        return false;
    // largest image coordinate formed in the gather must stay in int32 (a
    // negative pre-padding starts the windows inside the image)
    const int64_t in_h = g.pad_h < 0 ? -g.pad_h : 0, in_w = g.pad_w < 0 ? -g.pad_w : 0;
    if ((g.P - 1) * g.str_h + (g.R - 1) * g.dil_h + in_h >= lim ||
        (g.Q - 1) * g.str_w + (g.S - 1) * g.dil_w + in_w >= lim)
        return false;
    if (g.R * g.S > (1 << 20)) return false;
    return true;
}

// Whether the NCHW-row variants can read the image in place: each channel's
// rows contiguous with 16-byte aligned strides (the 4-D TMA map), rows of W
// bytes with W a multiple of 16 and at most 192, and every k-step's pixels
// whole 4-byte runs of image rows: stride 1 along W, Q, pre-padding along W
// and the tap offsets s*dil_w all multiples of 4.  The image rows one
// 128-pixel tile lies on must fit one staging slot: a tile starts at column
// q0 = 128t mod Q, a multiple of gcd(128, Q), so it spans at most
// (Q - gcd(128, Q) + 127) / Q + 1 rows.
static bool nchw_rows_fit(const ConvGeom &g, const void *x_dev) {
    if (g.W % 16 != 0 || g.W > NCHW_MAX_ROW_BYTES) return false;
    if (g.xs[3] != 1 || g.xs[2] % 16 != 0 || g.xs[1] % 16 != 0 || g.xs[0] % 16 != 0) return false;
    if (x_dev != nullptr && ((uintptr_t)x_dev % 16) != 0) return false;
    if (g.xs[0] >= ((int64_t)1 << 40) || g.xs[1] >= ((int64_t)1 << 40) || g.xs[2] >= ((int64_t)1 << 40)) return false;
    if (g.H >= ((int64_t)1 << 31) || g.N >= ((int64_t)1 << 31) || g.C >= ((int64_t)1 << 31)) return false;
    if (g.str_w != 1 || g.Q % 4 != 0 || g.pad_w % 4 != 0 || (g.S > 1 && g.dil_w % 4 != 0)) return false;
    const int64_t gq = std::gcd((int64_t)MT, g.Q);
    const int64_t rows = (g.Q - gq + MT - 1) / g.Q + 1;
    return rows * g.W <= NCHW_MAX_ROW_BYTES;
}

void igemm_plan(const ConvGeom &g, const void *x_dev, IgemmPlan *pl, bool register_loads, bool nchw_rows_ok) {
    const bool direct = g.xs[1] == 1 && (g.C % 16) == 0 && (g.xs[0] % 16) == 0 && (g.xs[2] % 16) == 0 &&
                        (g.xs[3] % 16) == 0 && (x_dev == nullptr || ((uintptr_t)x_dev % 16) == 0);
    // output channels per tile: 128, 192 or 256 (the smallest that covers
    // K, so that no MMA column is wasted on 129..192 channels)
    pl->n_tile = g.K > 192 ? 256 : (g.K > 128 ? 192 : 128);
    // an image that is not channels-last is read in place by the NCHW-row
    // variants (128- and 192-column tiles) where they fit, else copied to
    // channels-last first
    pl->nchw_rows = !direct && !register_loads && nchw_rows_ok && pl->n_tile <= 192 && nchw_rows_fit(g, x_dev);
    pl->pack_x = !direct && !pl->nchw_rows;
    pl->pack_done = false;
    pl->register_loads = register_loads;
    pl->c16 = (g.C + 15) / 16 * 16;
    pl->c_steps = (g.C + KS - 1) / KS;
    pl->k_steps = g.R * g.S * pl->c_steps;
    pl->n_tiles = (g.K + pl->n_tile - 1) / pl->n_tile;
    pl->m_tiles = (g.N * g.P * g.Q + MT - 1) / MT;
    pl->wpack_bytes = (size_t)align256(pl->n_tiles * pl->k_steps * pl->n_tile * (int64_t)(KS * 2));
    // one tile of output channels whose filter blocks fit in shared memory:
    // the filter stays resident in every CTA (taken with the TMA producers)
    // (256-column tiles: the 128- and 192-column ones put their image tile
    // in tensor memory and spend the shared memory on image staging instead)
    pl->resident_b =
        pl->n_tile == 256 && pl->n_tiles == 1 && pl->k_steps * pl->n_tile * (int64_t)(KS * 2) <= RESB_MAX_BYTES;
    // the image copy keeps only the rows the windows read: with
    // g = gcd(stride_h, dilation_h) (stride_h for a one-row filter) every
    // row read is h = p*stride_h - pre_h + r*dil_h = -pre_h (mod g)
    pl->row0 = 0;
    pl->row_step = 1;
    pl->hp = g.H;
    if (pl->pack_x) {
        int64_t gh = g.R > 1 ? std::gcd(g.str_h, g.dil_h) : g.str_h;
        if (gh > 1) {
            const int64_t r0 = ((-g.pad_h) % gh + gh) % gh;
            const int64_t hp = g.H > r0 ? (g.H - r0 + gh - 1) / gh : 0;
            if (hp >= 1) {
                pl->row0 = r0;
                pl->row_step = gh;
                pl->hp = hp;
            }
        }
    }
    pl->xpack_bytes = pl->pack_x ? (size_t)align256(g.N * pl->hp * g.W * pl->c16) : 0;
    // One CTA per SM walks the tiles.  With fewer tiles than SMs and long
    // reductions (the weight gradient's shape: few output tiles, a reduction
    // over every pixel of the batch) the tiles are cut along the reduction
    // into as many runs as keep the SMs busy, each at least kMinSplitSteps
    // long; the reduction kernel adds the runs' int32 sums and finishes the
    // tiles.
    // With more tiles than SMs and a short partial last round (rem tiles, at
    // most a quarter of the SMs), the tiles of that round are cut the same
    // way into runs of at least kMinTailSteps k-steps: the round takes a
    // fraction of a tile's time instead of a whole one.  (Longer last rounds
    // were measured too: the reduction of their runs costs more than it
    // saves.)
    const int64_t tiles = pl->m_tiles * pl->n_tiles;
    const int64_t sms = device_sm_count();
    pl->splits = 1;
    int64_t cut_tiles = 0;
    if (tiles > 0 && tiles < sms && pl->k_steps >= kSplitMinKSteps) {
        int64_t sp = sms / tiles;
        if (sp > pl->k_steps / kMinSplitSteps) sp = pl->k_steps / kMinSplitSteps;
        if (sp > kMaxSplits) sp = kMaxSplits;
        if (sp >= 2) {
            pl->splits = sp;
            cut_tiles = tiles;
        }
    } else if (tiles > sms && tiles % sms != 0 && tiles % sms <= sms / 4 && pl->k_steps >= 4 * kMinTailSteps) {
        const int64_t rem = tiles % sms;
        int64_t sp = sms / rem;
        if (sp > pl->k_steps / kMinTailSteps) sp = pl->k_steps / kMinTailSteps;
        if (sp > kMaxSplits) sp = kMaxSplits;
        if (sp >= 4) {
            pl->splits = sp;
            cut_tiles = rem;
        }
    }
    pl->full_units = tiles - cut_tiles;
    pl->num_units = pl->full_units + cut_tiles * pl->splits;
    pl->grid = pl->num_units < sms ? pl->num_units : sms;
    // workspace: [filter blocks][partial sums][image copy]
    size_t off = pl->wpack_bytes;
    pl->tail_part_off = off;
    pl->tail_part_bytes = 0;
    if (pl->splits > 1) {
        pl->tail_part_bytes = (size_t)align256(cut_tiles * pl->splits * MT * pl->n_tile * 4);
        off += pl->tail_part_bytes;
    }
    pl->xpack_off = off;
    pl->workspace_bytes = off + pl->xpack_bytes;
}

bool igemm_filter_in_kernel(const ConvGeom &g, const IgemmPlan &pl, const void *w) {
    const int64_t lim40 = (int64_t)1 << 40, lim32 = (int64_t)1 << 32;
    // (the image taken by TMA: the im2col limits; a pixel-row map, where a
    // 1x1 call takes one, has none of its own)
    return pl.n_tile <= 192 && !pl.register_loads && !pl.nchw_rows && im2col_geometry_ok(kernel_geom(g, pl)) &&
           g.ws[1] == 1 && g.ws[3] % 16 == 0 &&
           g.ws[2] % 16 == 0 && g.ws[0] % 16 == 0 && g.ws[0] < lim40 && g.ws[2] < lim40 && g.ws[3] < lim40 &&
           g.C < lim32 && g.K < lim32 && (w == nullptr || ((uintptr_t)w % 16) == 0);
}

static PackFilterJob pack_job(const ConvGeom &g, const IgemmPlan &pl, const int8_t *w, uint8_t *wp) {
    PackFilterJob j;
    j.w = w;
    j.ws0 = g.ws[0];
    j.ws1 = g.ws[1];
    j.ws2 = g.ws[2];
    j.ws3 = g.ws[3];
    j.K = (int32_t)g.K;
    j.C = (int32_t)g.C;
    j.R = (int32_t)g.R;
    j.S = (int32_t)g.S;
    j.mode = g.mode;
    j.c_steps = (int32_t)pl.c_steps;
    j.k_steps = (int32_t)pl.k_steps;
    j.n_tiles = (int32_t)pl.n_tiles;
    j.nt_rows = (int32_t)pl.n_tile;
    j.kperm = pl.nchw_rows ? 1 : 0;
    j.fd_rows = make_fastdiv(pl.n_tile);
    j.fd_ksteps = make_fastdiv(pl.k_steps);
    j.fd_csteps = make_fastdiv(pl.c_steps);
    j.fd_s = make_fastdiv(g.S);
    j.wp = wp;
    return j;
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
    if (!pl.nchw_rows && (g.K == 1 || g.ws[0] == 1) && g.ws[1] % 16 == 0 && g.ws[2] % 16 == 0 && g.ws[3] % 16 == 0 &&
        ((uintptr_t)w % 16) == 0) {
        // output channels adjacent: the transposing repack
        const int64_t tb = pl.n_tiles * pl.k_steps * (pl.n_tile / 64);
        igemm_pack_filter_k_minor_kernel<<<(unsigned)(tb < (int64_t)sms * 16 ? tb : (int64_t)sms * 16), 256, 0, st>>>(
            pack_job(g, pl, w, wp));
    } else if (total >= ((int64_t)1 << 31))
        igemm_pack_filter_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(pack_job(g, pl, w, wp));
    else
        igemm_pack_filter_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(pack_job(g, pl, w, wp));
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

conv_status igemm_wgrad_fold_launch(const WgradFold &fd, const IgemmPlan &pl, int8_t *x2, void *workspace,
                                    void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    WgradFoldArgs f;
    std::memset(&f, 0, sizeof(f));
    f.x = fd.x; f.xs0 = fd.xs[0]; f.xs1 = fd.xs[1]; f.xs2 = fd.xs[2]; f.xs3 = fd.xs[3];
    f.dy = fd.dy; f.ys0 = fd.ys[0]; f.ys1 = fd.ys[1]; f.ys2 = fd.ys[2]; f.ys3 = fd.ys[3];
    f.N = fd.N; f.C = fd.C; f.H = fd.H; f.W = fd.W; f.K = fd.K; f.P = fd.P; f.Q = fd.Q;
    f.T = fd.T; f.Q2 = fd.Q2; f.U = fd.U; f.c16 = fd.c16; f.pre_w = fd.pre_w; f.stride_w = fd.stride_w;
    // 16-byte loads of 16 consecutive images (channels of X) or rows (K of dY)
    f.x_vec = (fd.C == 1 || fd.xs[1] == 1) && fd.xs[0] % 16 == 0 && fd.xs[2] % 16 == 0 && fd.xs[3] % 16 == 0 &&
                      ((uintptr_t)fd.x % 16) == 0
                  ? 1
                  : 0;
    f.dy_vec = (fd.K == 1 || fd.ys[1] == 1) && fd.ys[0] % 16 == 0 && fd.ys[2] % 16 == 0 && fd.ys[3] % 16 == 0 &&
                       ((uintptr_t)fd.dy % 16) == 0
                   ? 1
                   : 0;
    f.nt_rows = (int32_t)pl.n_tile;
    f.n_tiles = (int32_t)pl.n_tiles;
    f.k_steps = (int32_t)pl.k_steps;
    f.x2 = x2;
    f.wp = static_cast<uint8_t *>(workspace);
    const int64_t xb = ((fd.C + 63) / 64) * fd.H * fd.U;
    const int64_t wb = pl.n_tiles * pl.k_steps * (pl.n_tile / 64);
    if (xb > 0)
        igemm_wgrad_fold_image_kernel<<<(unsigned)(xb < (int64_t)sms * 16 ? xb : (int64_t)sms * 16), 256, 0, st>>>(f);
    if (wb > 0)
        igemm_wgrad_fold_filter_kernel<<<(unsigned)(wb < (int64_t)sms * 16 ? wb : (int64_t)sms * 16), 256, 0, st>>>(
            f);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

conv_status igemm_pack_filter_group_launch(int n, const ConvGeom *const *g, const IgemmPlan *const *pl,
                                           const int8_t *const *w, void *const *workspace, void *stream) {
    if (n < 1 || n > kMaxPackJobs) return CONV_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    PackFilterJobs js;
    std::memset(&js, 0, sizeof(js));
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        js.job[i] = pack_job(*g[i], *pl[i], w[i], static_cast<uint8_t *>(workspace[i]));
        total += pl[i]->n_tiles * pl[i]->k_steps * pl[i]->n_tile * 8;
        js.end[i] = total;
    }
    js.n = n;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    if (blocks == 0) return CONV_OK;
    if (total >= ((int64_t)1 << 31))
        igemm_pack_filter_group_kernel<true><<<(unsigned)blocks, 256, 0, st>>>(js);
    else
        igemm_pack_filter_group_kernel<false><<<(unsigned)blocks, 256, 0, st>>>(js);
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

namespace {

PFN_cuTensorMapReplaceAddress_v12000 address_replacer() {
    static std::atomic<void *> fn{nullptr};
    static std::atomic<bool> tried{false};
    if (!tried.load()) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapReplaceAddress", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn.store(p);
        tried.store(true);
    }
    return reinterpret_cast<PFN_cuTensorMapReplaceAddress_v12000>(fn.load());
}

enum Variant {
    V_REG128, V_REG192, V_REG256, V_TMEM128, V_TMEM192, V_TMA256, V_RESB256, V_NCHW128, V_NCHW192, V_SELF128, V_SELF192
};

// Everything a launch of the convolution kernel needs that does not change
// with the buffers' addresses: the kernel arguments (tensor maps encoded for
// the addresses of the call that built them) and the kernel variant.
struct LaunchPlan {
    IgemmArgs a;
    int variant;
    bool tma;
    bool planes;          // plane-contiguous image copy (when the image is repacked)
    const void *x_map;    // addresses the maps were encoded with
    const void *y_map;
    const void *w_map;    // (filter map: in-kernel filter conversion only)
};

// Launch-plan cache: key = geometry, plan, device and the 16-byte alignment
// of the image and output pointers; a hit re-targets the cached tensor maps
// to the call's addresses with cuTensorMapReplaceAddress instead of encoding
// them again.  Least recently used entries give way; conv_shutdown empties it.
struct LaunchKey {
    int64_t v[64];
    int n;
};

// The key's fields, one int64 each (no padding bytes compared).
LaunchKey make_key(const ConvGeom &g, const IgemmPlan &pl, int dev, int align) {
    LaunchKey k;
    std::memset(&k, 0, sizeof(k));
    int n = 0;
    auto put = [&](int64_t v) { k.v[n++] = v; };
    put(g.N); put(g.C); put(g.H); put(g.W); put(g.K); put(g.R); put(g.S); put(g.P); put(g.Q);
    for (int i = 0; i < 4; ++i) { put(g.xs[i]); put(g.ws[i]); put(g.ys[i]); }
    put(g.pad_h); put(g.pad_w); put(g.str_h); put(g.str_w); put(g.dil_h); put(g.dil_w);
    put(g.mode); put(g.bias); put(g.relu); put(g.out_int8); put(g.out_shift);
    put(pl.pack_x); put(pl.nchw_rows); put(pl.register_loads); put(pl.resident_b); put(pl.n_tile); put(pl.c16); put(pl.c_steps);
    put(pl.k_steps); put(pl.n_tiles); put(pl.m_tiles); put((int64_t)pl.wpack_bytes); put((int64_t)pl.xpack_bytes);
    put(pl.full_units); put(pl.splits); put(pl.num_units); put(pl.grid); put((int64_t)pl.tail_part_off);
    put((int64_t)pl.tail_part_bytes); put((int64_t)pl.xpack_off); put((int64_t)pl.workspace_bytes);
    put(pl.row0); put(pl.row_step); put(pl.hp);
    put(dev); put(align);
    k.n = n;
    return k;
}

constexpr int kLaunchCacheSize = 32;
struct LaunchCacheEntry {
    LaunchKey key;
    LaunchPlan plan;
    uint64_t used;
    bool valid;
};
std::mutex g_launch_mu;
LaunchCacheEntry g_launch_cache[kLaunchCacheSize];
uint64_t g_launch_clock = 0;
std::atomic<uint64_t> g_launch_hits{0}, g_launch_misses{0};

bool launch_lookup(const LaunchKey &k, LaunchPlan *out) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    for (auto &e : g_launch_cache)
        if (e.valid && std::memcmp(&e.key, &k, sizeof(k)) == 0) {
            e.used = ++g_launch_clock;
            *out = e.plan;
            return true;
        }
    return false;
}

void launch_insert(const LaunchKey &k, const LaunchPlan &p) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    LaunchCacheEntry *victim = &g_launch_cache[0];
    for (auto &e : g_launch_cache) {
        if (!e.valid) {
            victim = &e;
            break;
        }
        if (e.used < victim->used) victim = &e;
    }
    victim->key = k;
    victim->plan = p;
    victim->used = ++g_launch_clock;
    victim->valid = true;
}


// Builds the launch plan of a call (kernel arguments, tensor maps, variant).
// The channels-last copy of the image takes the plane transpose: each
// channel's rows contiguous, whole 16-byte loads inside a row when rows are
// skipped.
bool planes_copy(const ConvGeom &g0, const IgemmPlan &pl, const int8_t *x) {
    const int64_t hw = g0.H * g0.W;
    return (g0.W == 1 || g0.xs[3] == 1) && (g0.H == 1 || g0.xs[2] == g0.W) && g0.xs[1] % 16 == 0 &&
           g0.xs[0] % 16 == 0 && hw % 16 == 0 && ((uintptr_t)x % 16) == 0 && hw < ((int64_t)1 << 31) &&
           (pl.row_step == 1 || g0.W % 16 == 0);
}

// Whether the image's images are adjacent bytes (batch stride 1, as in the
// weight gradient's exchanged view of a channels-last image) with 16-byte
// aligned channel and pixel strides and base: igemm_pack_image_batch_minor_kernel.
bool batch_minor_copy(const ConvGeom &g0, const int8_t *x) {
    return (g0.N == 1 || g0.xs[0] == 1) && g0.xs[1] % 16 == 0 && g0.xs[2] % 16 == 0 && g0.xs[3] % 16 == 0 &&
           ((uintptr_t)x % 16) == 0 && g0.H * g0.W < ((int64_t)1 << 31);
}

// 4-D map {C, S, R, K} of an int8 filter with contiguous channels (byte
// strides ws[3], ws[2], ws[0]): box {64, 1, 1, NT}, the k-step's int8 tile,
// no swizzle (the converters read 64-byte rows).
bool encode_filter_map(const ConvGeom &g, const void *w, int64_t nt, CUtensorMap *map) {
    auto enc = tiled_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)g.C, (cuuint64_t)g.S, (cuuint64_t)g.R, (cuuint64_t)g.K};
    const cuuint64_t strides[3] = {(cuuint64_t)g.ws[3], (cuuint64_t)g.ws[2], (cuuint64_t)g.ws[0]};
    const cuuint32_t box[4] = {(cuuint32_t)KS, 1, 1, (cuuint32_t)nt};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(w), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

conv_status build_launch(const ConvGeom &g0, const IgemmPlan &pl, const int8_t *x, const int8_t *w, void *y,
                         uint8_t *wp, LaunchPlan *L) {
    const ConvGeom g = kernel_geom(g0, pl);
    IgemmArgs &a = L->a;
    std::memset(&a, 0, sizeof(a));
    L->planes = false;
    if (pl.pack_x) {
        L->planes = planes_copy(g0, pl, x);
        a.x = reinterpret_cast<int8_t *>(wp + pl.xpack_off);
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
    a.out_int8 = g.out_int8 ? 1 : 0;
    a.out_shift = g.out_shift;
    a.ys_n = g.ys[0]; a.ys_k = g.ys[1]; a.ys_p = g.ys[2]; a.ys_q = g.ys[3];
    a.H = (int32_t)g.H; a.W = (int32_t)g.W; a.P = (int32_t)g.P; a.Q = (int32_t)g.Q;
    a.K = (int32_t)g.K; a.S = (int32_t)g.S;
    a.c16 = (int32_t)pl.c16;
    a.c_steps = (int32_t)pl.c_steps;
    a.k_steps = (int32_t)pl.k_steps;
    a.pad_h = (int32_t)g.pad_h; a.pad_w = (int32_t)g.pad_w;
    a.str_h = (int32_t)g.str_h; a.str_w = (int32_t)g.str_w;
    a.dil_h = (int32_t)g.dil_h; a.dil_w = (int32_t)g.dil_w;
    a.m_total = (int32_t)(g.N * g.P * g.Q);
    a.n_tiles = (int32_t)pl.n_tiles;
    a.fd_nt = make_fastdiv(pl.n_tiles);
    a.fd_pq = make_fastdiv(g.P * g.Q);
    a.fd_q = make_fastdiv(g.Q);
    a.fd_cs = make_fastdiv(pl.c_steps);
    a.fd_s = make_fastdiv(g.S);
    a.num_tiles = (int32_t)(pl.m_tiles * pl.n_tiles);
    a.full_units = (int32_t)pl.full_units;
    a.splits = (int32_t)pl.splits;
    a.num_units = (int32_t)pl.num_units;
    a.tail_part = pl.splits > 1 ? reinterpret_cast<int32_t *>(wp + pl.tail_part_off) : nullptr;
    a.relu = g.relu ? 1 : 0;
    a.y_vec = (!g.out_int8 && g.ys[1] == 1 && (g.K % 4) == 0 && ((uintptr_t)y % 16) == 0 && (g.ys[0] % 4) == 0 &&
               (g.ys[2] % 4) == 0 && (g.ys[3] % 4) == 0)
                  ? 1
                  : 0;
    a.wait_limit_ns = wait_limit_ns();
    a.status = device_status_word();
    if (!a.status) return CONV_ERR_CUDA;
    // a 1x1 filter at stride 1 without padding over dense pixel rows reads
    // image pixel m for output pixel m: plain 2-D boxes instead of im2col
    const int64_t c_dim = pl.pack_x ? pl.c16 : g.C;
    a.a_rows = (!pl.nchw_rows && g.R == 1 && g.S == 1 && g.str_h == 1 && g.str_w == 1 && g.pad_h == 0 && g.pad_w == 0 &&
                g.P == g.H && g.Q == g.W && a.xs_h == g.W * a.xs_w && a.xs_n == g.H * a.xs_h)
                   ? 1
                   : 0;
    // 128- and 192-column tiles keep the f16 image tile in tensor memory;
    // their staging loads are 64-byte swizzled for the converters' row reads
    const bool tmem_a = pl.n_tile <= 192;
    bool tma = false;
    if (pl.nchw_rows) {
        // the planner checked everything the map needs
        if (!encode_nchw_rows_map(g, x, &a.tmap_x)) return CONV_ERR_CUDA;
        tma = true;
    } else if (!pl.register_loads) {
        if (a.a_rows) tma = encode_rows_map(g, a.x, a.xs_w, c_dim, tmem_a, &a.tmap_x);
        if (!tma) {
            a.a_rows = 0;
            tma = encode_im2col_map(g, a.x, a.xs_n, a.xs_h, a.xs_w, c_dim, tmem_a, &a.tmap_x);
        }
    }
    // tensor-memory tiles over a channels-last image convert a channel-
    // contiguous filter themselves (no repack launch)
    a.R = (int32_t)g.R;
    a.mode = g.mode;
    const bool self_b = w != nullptr && tma && tmem_a && !pl.nchw_rows && igemm_filter_in_kernel(g0, pl, w) &&
                        encode_filter_map(g0, w, pl.n_tile, &a.tmap_w);
    L->w_map = self_b ? w : nullptr;
    // the 128-column tensor-memory variant stages 32 output columns per store
    // (16 when the kernel also converts the filter)
    const bool wide_out = tma && pl.n_tile == 128 && !self_b;
    a.y_tma = encode_output_map(g, y, wide_out, &a.tmap_y) ? 1 : (encode_output_map_nchw(g, y, wide_out, &a.tmap_y) ? 2 : 0);
    // int8 outputs are staged 64 columns at a time: a 192-column tile (96
    // per epilogue warp) stores them with plain stores
    if (g.out_int8 && pl.n_tile == 192) a.y_tma = 0;
    // TMA path: 128- and 192-column tiles keep the image tile in tensor
    // memory; 256-column tiles keep it in shared memory, with the filter
    // resident when it fits
    L->tma = tma;
    if (pl.nchw_rows)
        L->variant = pl.n_tile == 128 ? V_NCHW128 : V_NCHW192;
    else if (self_b)
        L->variant = pl.n_tile == 128 ? V_SELF128 : V_SELF192;
    else if (tma && tmem_a)
        L->variant = pl.n_tile == 128 ? V_TMEM128 : V_TMEM192;
    else if (tma && pl.resident_b)
        L->variant = V_RESB256;
    else if (tma)
        L->variant = V_TMA256;
    else
        L->variant = pl.n_tile == 256 ? V_REG256 : (pl.n_tile == 192 ? V_REG192 : V_REG128);
    L->x_map = a.x;
    L->y_map = y;
    return CONV_OK;
}

}  // namespace

void igemm_cache_clear() {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    for (auto &e : g_launch_cache) e.valid = false;
}

void igemm_cache_stats(uint64_t *hits, uint64_t *misses) {
    *hits = g_launch_hits.load();
    *misses = g_launch_misses.load();
}

conv_status igemm_pack_image_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, void *workspace,
                                    void *stream) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    int8_t *xp = reinterpret_cast<int8_t *>(wp + pl.xpack_off);
    const int64_t hwp = pl.hp * g.W;  // pixels of each copied image
    if (g.N * hwp == 0) return CONV_OK;
    if (planes_copy(g, pl, x)) {
        const int64_t total = g.N * ((hwp + kPackPix - 1) / kPackPix) * ((pl.c16 + kPackCh - 1) / kPackCh);
        int64_t blocks = total < (int64_t)sms * 8 ? total : (int64_t)sms * 8;
        igemm_pack_image_planes_kernel<<<(unsigned)blocks, 256, 0, st>>>(
            x, g.xs[0], g.xs[1], g.N, (int32_t)g.C, (int32_t)hwp, (int32_t)g.W, (int32_t)pl.row0,
            (int32_t)pl.row_step, (int32_t)pl.c16, xp);
    } else if (batch_minor_copy(g, x)) {
        const int64_t total = ((g.N + 63) / 64) * hwp * ((pl.c16 + 63) / 64);
        const int64_t blocks = total < (int64_t)sms * 16 ? total : (int64_t)sms * 16;
        igemm_pack_image_batch_minor_kernel<<<(unsigned)blocks, 256, 0, st>>>(
            x, g.xs[1], g.xs[2], g.xs[3], g.N, (int32_t)g.C, (int32_t)pl.hp, (int32_t)g.W, (int32_t)pl.row0,
            (int32_t)pl.row_step, (int32_t)pl.c16, xp);
    } else {
        const int64_t total = g.N * pl.hp * g.W * (pl.c16 / 16);
        int64_t blocks = (total + 255) / 256;
        if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
        igemm_pack_image_kernel<<<(unsigned)blocks, 256, 0, st>>>(x, g.xs[0], g.xs[1], g.xs[2], g.xs[3], g.N,
                                                                  (int32_t)g.C, (int32_t)pl.hp, (int32_t)g.W,
                                                                  (int32_t)pl.row0, (int32_t)pl.row_step,
                                                                  (int32_t)pl.c16, xp);
    }
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

namespace {

// The launch plan of a call (variant, grid, arguments with their tensor
// maps): from the cache when an equal call ran before, re-targeted to this
// call's buffers.
conv_status prepare_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, const int8_t *w, void *y,
                           const int32_t *bias, uint8_t *wp, LaunchPlan *out) {
    int dev = 0;
    cudaGetDevice(&dev);
    // (every decision of build_launch that reads a pointer reads only its
    // 16-byte alignment, or, for the filter, whether it is given)
    const int walign = w == nullptr ? 0 : (((uintptr_t)w % 16) == 0 ? 4 : 8);
    const LaunchKey key =
        make_key(g, pl, dev, (((uintptr_t)x % 16) == 0 ? 1 : 0) | (((uintptr_t)y % 16) == 0 ? 2 : 0) | walign);
    LaunchPlan L;
    bool hit = launch_lookup(key, &L);
    const void *x_now = pl.pack_x ? (const void *)(wp + pl.xpack_off) : (const void *)x;
    if (hit && (L.x_map != x_now || L.y_map != y || (L.w_map && L.w_map != w))) {
        // re-target the cached maps to this call's buffers
        auto rep = address_replacer();
        bool ok = rep != nullptr;
        if (ok && L.tma && L.x_map != x_now) ok = rep(&L.a.tmap_x, const_cast<void *>(x_now)) == CUDA_SUCCESS;
        if (ok && L.a.y_tma && L.y_map != y) ok = rep(&L.a.tmap_y, y) == CUDA_SUCCESS;
        if (ok && L.w_map && L.w_map != w) ok = rep(&L.a.tmap_w, const_cast<int8_t *>(w)) == CUDA_SUCCESS;
        hit = ok;
    }
    if (hit) {
        g_launch_hits.fetch_add(1);
        L.a.x = static_cast<const int8_t *>(x_now);
        L.a.y = y;
        L.a.wp = wp;
        L.a.tail_part = pl.splits > 1 ? reinterpret_cast<int32_t *>(wp + pl.tail_part_off) : nullptr;
        L.x_map = x_now;
        L.y_map = y;
        if (L.w_map) L.w_map = w;
    } else {
        g_launch_misses.fetch_add(1);
        conv_status b = build_launch(g, pl, x, w, y, wp, &L);
        if (b) return b;
        launch_insert(key, L);
    }
    L.a.bias = g.bias ? bias : nullptr;
    *out = L;
    return CONV_OK;
}

template <int NT, bool kTma, bool kResB = false, bool kTmemA = false, bool kNchw = false>
conv_status launch_conv_group(const IgemmGroup &grp, int grid, cudaStream_t st) {
    using Cfg = TileCfg<NT, kTma, kResB, kTmemA, kNchw, false>;
    static std::atomic<bool> attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev].load()) {
        if (cudaFuncSetAttribute(igemm_conv_group_kernel<NT, kTma, kResB, kTmemA, kNchw, false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess)
            return CONV_ERR_CUDA;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, igemm_conv_group_kernel<NT, kTma, kResB, kTmemA, kNchw, false>, grp) != cudaSuccess)
        return CONV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // namespace

conv_status igemm_group_launch(int n, const ConvGeom *const *g, const IgemmPlan *const *pl, const int8_t *x,
                               void *const *y, void *const *workspace, void *stream, bool *launched,
                               bool after_own_repack) {
    *launched = false;
    if (n < 2 || n > kMaxGroup) return CONV_OK;
    static IgemmGroup grp_zero;  // (zero-filled template: IgemmArgs has no constructor)
    IgemmGroup grp = grp_zero;
    int variant = -1;
    for (int c = 0; c < n; ++c) {
        // whole tiles only (no reduction kernel), and the image copy, if
        // any, already made by the caller
        if (pl[c]->splits > 1 || (pl[c]->pack_x && !pl[c]->pack_done) || pl[c]->m_tiles * pl[c]->n_tiles == 0)
            return CONV_OK;
        LaunchPlan L;
        conv_status st = prepare_launch(*g[c], *pl[c], x, nullptr, y[c], nullptr, static_cast<uint8_t *>(workspace[c]), &L);
        if (st) return st;
        if (!(L.variant == V_TMEM128 || L.variant == V_TMEM192 || L.variant == V_TMA256 || L.variant == V_RESB256 ||
              L.variant == V_NCHW128 || L.variant == V_NCHW192) ||
            (variant >= 0 && L.variant != variant))
            return CONV_OK;
        variant = L.variant;
        grp.cls[c] = L.a;
        grp.cls[c].early_image = after_own_repack && L.tma ? 1 : 0;
    }
    // CTAs per convolution, together at most one per SM: each CTA walks its
    // convolution's tiles, a tile costing its k-steps plus about kEpiSteps
    // k-steps of set-up and epilogue (which dominate the one- and two-tap
    // classes of a strided data gradient).  Starting from one CTA each, every
    // further SM goes to the convolution whose CTAs finish last
    // (ceil(tiles / CTAs) x cost per tile) while it has a tile without a CTA.
    constexpr int64_t kEpiSteps = 5;
    const int sms = device_sm_count();
    int cta[kMaxGroup];
    int used = n;
    for (int c = 0; c < n; ++c) cta[c] = 1;
    auto span = [&](int c) {
        return (pl[c]->num_units + cta[c] - 1) / cta[c] * (pl[c]->k_steps + kEpiSteps);
    };
    while (used < sms) {
        int best = -1;
        for (int c = 0; c < n; ++c)
            if (cta[c] < pl[c]->num_units && (best < 0 || span(c) > span(best))) best = c;
        if (best < 0) break;
        ++cta[best];
        ++used;
    }
    grp.n = n;
    grp.cta_start[0] = 0;
    for (int c = 0; c < n; ++c) grp.cta_start[c + 1] = grp.cta_start[c] + cta[c];
    cudaStream_t st = (cudaStream_t)stream;
    conv_status rc;
    switch (variant) {
        case V_TMEM128: rc = launch_conv_group<128, true, false, true>(grp, used, st); break;
        case V_TMEM192: rc = launch_conv_group<192, true, false, true>(grp, used, st); break;
        case V_TMA256: rc = launch_conv_group<256, true>(grp, used, st); break;
        case V_NCHW128: rc = launch_conv_group<128, true, false, true, true>(grp, used, st); break;
        case V_NCHW192: rc = launch_conv_group<192, true, false, true, true>(grp, used, st); break;
        default: rc = launch_conv_group<256, true, true>(grp, used, st); break;
    }
    if (rc == CONV_OK) *launched = true;
    return rc;
}

conv_status igemm_main_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, const int8_t *w, void *y,
                              const int32_t *bias, void *workspace, void *stream, bool repack) {
    cudaStream_t st = (cudaStream_t)stream;
    const int sms = device_sm_count();
    uint8_t *wp = static_cast<uint8_t *>(workspace);
    if (pl.m_tiles * pl.n_tiles == 0) return CONV_OK;
    LaunchPlan L;
    // a call that brings its filter (repack) may have the kernel convert it
    // itself; a call on a repacked workspace reads the repacked blocks
    conv_status pst = prepare_launch(g, pl, x, repack ? w : nullptr, y, bias, wp, &L);
    if (pst) return pst;
    IgemmArgs &a = L.a;
    const bool self_b = L.variant == V_SELF128 || L.variant == V_SELF192;
    // the filter repack, unless the kernel converts the filter itself
    const bool repacked = repack && !self_b;
    if (repacked && (pst = igemm_pack_filter_launch(g, pl, w, workspace, stream))) return pst;
    // the image loads may start before the filter repack ends only when the
    // repack is the kernel right before (not an image copy, whose output
    // they read)
    a.early_image = repacked && L.tma && !(pl.pack_x && !pl.pack_done) ? 1 : 0;
    if (pl.pack_x && !pl.pack_done) {
        const conv_status pr = igemm_pack_image_launch(g, pl, x, workspace, stream);
        if (pr) return pr;
    }
    const int grid = (int)pl.grid;
    conv_status rc;
    switch (L.variant) {
        case V_TMEM128: rc = launch_conv<128, true, false, true>(a, grid, st); break;
        case V_RESB256: rc = launch_conv<256, true, true>(a, grid, st); break;
        case V_TMA256: rc = launch_conv<256, true>(a, grid, st); break;
        case V_TMEM192: rc = launch_conv<192, true, false, true>(a, grid, st); break;
        case V_NCHW128: rc = launch_conv<128, true, false, true, true>(a, grid, st); break;
        case V_NCHW192: rc = launch_conv<192, true, false, true, true>(a, grid, st); break;
        case V_SELF128: rc = launch_conv<128, true, false, true, false, true>(a, grid, st); break;
        case V_SELF192: rc = launch_conv<192, true, false, true, false, true>(a, grid, st); break;
        case V_REG256: rc = launch_conv<256, false>(a, grid, st); break;
        case V_REG192: rc = launch_conv<192, false>(a, grid, st); break;
        default: rc = launch_conv<128, false>(a, grid, st); break;
    }
    if (rc || pl.splits <= 1) return rc;
    const int32_t cut_tiles = a.num_tiles - a.full_units;
    int64_t blocks = (int64_t)cut_tiles * (pl.n_tile / kRedCols) * (MT / kRedRows);
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, igemm_split_reduce_kernel, (const int32_t *)a.tail_part, a.full_units, cut_tiles,
                           a.splits, a.n_tiles, (int32_t)pl.n_tile, a.m_total, a.K, a.P, a.Q, a.ys_n, a.ys_k,
                           a.ys_p, a.ys_q, a.y, a.out_int8, a.out_shift, a.bias, a.relu) != cudaSuccess)
        return CONV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

}  // namespace i8c
