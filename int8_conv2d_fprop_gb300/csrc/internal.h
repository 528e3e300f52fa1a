// internal.h -- declarations shared by the translation units of libint8conv.
// Not part of the public ABI (that is include/int8conv.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include "int8conv.h"

namespace i8c {

// Geometry of one validated call, flattened for the launchers.
struct ConvGeom {
    int64_t N, C, H, W;        // image
    int64_t K, R, S;           // filter
    int64_t P, Q;              // output
    int64_t xs[4], ws[4], ys[4];  // element strides (logical order)
    int64_t pad_h, pad_w;      // pre-padding (post padding only changes P, Q)
    int64_t str_h, str_w;
    int64_t dil_h, dil_w;
    int32_t mode;              // 0 cross-correlation, 1 convolution
    bool bias, relu;
    bool out_int8;             // int8 output: rounding right shift then saturation
    int32_t out_shift;
};

#ifdef __CUDACC__
// int8 output of CONV_EPILOGUE_INT8_OUT: floor((v + 2^(shift-1)) / 2^shift)
// for shift > 0, then clamped to [-128, 127].  In 32-bit arithmetic without
// overflow: floor(v / 2^s) is the arithmetic shift v >> s, and adding half
// before flooring adds exactly the bit just below the cut, (v >> (s-1)) & 1.
__device__ __forceinline__ int8_t requant_i8(int32_t v, int32_t shift) {
    int32_t t = v;
    if (shift > 0) t = (v >> shift) + ((v >> (shift - 1)) & 1);
    t = t > 127 ? 127 : (t < -128 ? -128 : t);
    return (int8_t)t;
}
#endif

// Fill g from validated descriptors.
void make_geom(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
               const conv_fprop_params *p, ConvGeom *g);

// Validation of the gradient calls (descriptors, shapes, parameters, the
// int32 accumulator bound).
conv_status validate_dgrad(const conv_tensor_desc *dy, const conv_tensor_desc *w, const conv_tensor_desc *dx,
                           const conv_fprop_params *p);
conv_status validate_wgrad(const conv_tensor_desc *x, const conv_tensor_desc *dy, const conv_tensor_desc *dw,
                           const conv_fprop_params *p);

// [lo, hi) byte ranges of two buffers overlap?
inline bool overlaps(const void *a, uint64_t a_bytes, const void *b, uint64_t b_bytes) {
    if (!a || !b || a_bytes == 0 || b_bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

// Largest addressed element offset + 1 of a descriptor (0 if a dim is 0).
int64_t desc_extent_elems(const conv_tensor_desc *d);

// ---------------------------------------------------------------- igemm
// Tile shape of the tensor-core kernel: 128 output pixels x n_tile (128 or
// 256) output channels, reduction consumed 64 channels (one 128-byte row of
// f16) at a time.
constexpr int kIgemmMTile = 128;
constexpr int kIgemmKStep = 64;

struct IgemmPlan {
    bool pack_x;            // image must be copied to channels-last first
    bool nchw_rows;         // image read in place from its NCHW rows (128- and 192-column tiles)
    bool pack_done;         // ... and the copy at xpack_off is made by the caller (igemm_pack_image_launch)
    bool register_loads;    // gather the image with global loads, not TMA im2col
    bool resident_b;        // the whole repacked filter stays in shared memory (TMA path)
    int64_t n_tile;         // output channels per tile (128, 192 or 256)
    int64_t c16;            // channel count rounded up to 16 (valid load width)
    int64_t c_steps;        // ceil(C / 64)
    int64_t k_steps;        // R * S * c_steps
    int64_t n_tiles;        // ceil(K / kIgemmNTile)
    int64_t m_tiles;        // ceil(N*P*Q / kIgemmMTile)
    size_t wpack_bytes;     // repacked filter
    size_t xpack_bytes;     // channels-last image copy (0 if not needed)
    // Rows of the image copy: when the stride and the dilation along H share
    // a factor g, only the rows h = row0 (mod g) are ever read, and the copy
    // holds those (hp of them); the convolution then runs on it with stride,
    // dilation and pre-padding divided by g (row_step = g; 1: every row).
    int64_t row0, row_step, hp;
    // Work split: with few tiles and long reductions each tile, and with a
    // short partial last round of tiles each tile of that round, is cut into
    // `splits` runs of k-steps computed by different CTAs (splits == 1: whole
    // tiles, full_units == num_units == tiles).
    int64_t full_units, splits, num_units, grid;
    size_t tail_part_off, tail_part_bytes;  // int32 partial sums of the cut tiles
    size_t xpack_off;       // image copy, after the filter and the partial sums
    size_t workspace_bytes; // total, each part 256-byte aligned
};

// Key of a call's plan: the three descriptors, the parameters, the device
// and whether the image pointer is 16-byte aligned (nullptr counts as
// aligned); equal keys give equal plans.
struct PlanKey {
    int64_t v[64];
    int n;
};
PlanKey make_plan_key(const conv_tensor_desc *x, const conv_tensor_desc *w, const conv_tensor_desc *y,
                      const conv_fprop_params *p, const void *x_dev, int dev);
// Empties the data-gradient plan cache.
void dgrad_cache_clear();

bool igemm_supported(const ConvGeom &g);
// register_loads: gather the image with global loads; nchw_rows_ok: the
// NCHW-row variants may be chosen.
void igemm_plan(const ConvGeom &g, const void *x_dev, IgemmPlan *pl, bool register_loads = false,
                bool nchw_rows_ok = true);
// Repacks the filter into the first pl.wpack_bytes of the workspace.
conv_status igemm_pack_filter_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *w, void *workspace,
                                     void *stream);
// Repacks the filters of n (<= kMaxPackJobs) planned convolutions, each into
// its own workspace, in one launch.
constexpr int kMaxPackJobs = 8;
conv_status igemm_pack_filter_group_launch(int n, const ConvGeom *const *g, const IgemmPlan *const *pl,
                                           const int8_t *const *w, void *const *workspace, void *stream);
// Runs n (2..4) planned convolutions of one image x (each with its own
// filter part of the workspace and output y[c]) as one launch of the
// tensor-core kernel, each on its share of the SMs.  Sets *launched = false,
// launching nothing, when the convolutions cannot share a launch (different
// kernel variants, cut tiles, an image copy still to make, register loads);
// the caller then runs them one by one.  after_own_repack: the launch
// directly follows the caller's own filter repack on the stream (see
// igemm_main_launch).
constexpr int kIgemmMaxGroup = 4;
conv_status igemm_group_launch(int n, const ConvGeom *const *g, const IgemmPlan *const *pl, const int8_t *x,
                               void *const *y, void *const *workspace, void *stream, bool *launched,
                               bool after_own_repack = false);
// Makes the channels-last copy of the image at pl.xpack_off of the workspace.
conv_status igemm_pack_image_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, void *workspace,
                                    void *stream);
// Runs the convolution (copying the image to channels-last first when
// pl.pack_x).  repack: launch the filter repack into the workspace first,
// unless the kernel variant converts the filter itself
// (igemm_filter_in_kernel); without it the workspace's filter part must
// already be packed, and the kernel reads it.  When
// the repack is launched it directly precedes the convolution on the stream
// (an ordinary launch, which starts once every earlier kernel of the stream
// has completed), so the image is final and the kernel's image loads need
// not wait for the repack to end.
conv_status igemm_main_launch(const ConvGeom &g, const IgemmPlan &pl, const int8_t *x, const int8_t *w, void *y,
                              const int32_t *bias, void *workspace, void *stream, bool repack);
// The weight gradient folded over T output columns of dY (grad.cu): X'' is
// the image copy [C][H][U][c16] with X''[c][h][u][t*N + n] =
// X[n, c, h, u - pre_w + t*stride_w] (zero outside X and for channels from
// T*N on), and the folded loss gradient the filter [K][P][Q2][c16] with
// channel t*N + n of tap (p, q2) = dY[n, k, p, T*q2 + t] (zero for columns
// from Q on), repacked into the filter blocks of pl (the plan of the folded
// forward convolution: one channel step per tap).  Strides in elements
// (bytes).
struct WgradFold {
    const int8_t *x;
    int64_t xs[4];  // X [N][C][H][W]
    const int8_t *dy;
    int64_t ys[4];  // dY [N][K][P][Q]
    int64_t N, C, H, W, K, P, Q;
    int64_t T, Q2, U, c16;
    int64_t pre_w, stride_w;
};
// Launches the copy into x2 (c16 * C * H * U bytes) and the repack into the
// workspace's filter part.
conv_status igemm_wgrad_fold_launch(const WgradFold &f, const IgemmPlan &pl, int8_t *x2, void *workspace,
                                    void *stream);

// Whether the 128- and 192-column tensor-memory kernels convert this
// call's filter themselves (channels contiguous, 16-byte aligned strides and
// pointer; w == nullptr: a 16-byte aligned pointer assumed) instead of
// reading repacked blocks.
bool igemm_filter_in_kernel(const ConvGeom &g, const IgemmPlan &pl, const void *w);

// Launch-plan cache of the tensor-core kernel (tensor maps re-targeted to
// each call's buffers): empty it; read its hit and miss counts.
void igemm_cache_clear();
void igemm_cache_stats(uint64_t *hits, uint64_t *misses);

// ---------------------------------------------------------------- direct
bool dp4a_supported(const ConvGeom &g);
conv_status dp4a_launch(const ConvGeom &g, const int8_t *x, const int8_t *w, void *y,
                        const int32_t *bias, void *stream);
conv_status generic_launch(const ConvGeom &g, const int8_t *x, const int8_t *w, void *y,
                           const int32_t *bias, void *stream);

// Workspace bytes a call needs given the actual image pointer (a misaligned
// pointer needs the channels-last image copy too).
conv_status conv_fprop_workspace_size_for(const conv_tensor_desc *x, const void *x_dev, const conv_tensor_desc *w,
                                          const conv_tensor_desc *y, const conv_fprop_params *p, size_t *bytes);

// ---------------------------------------------------------------- device
// Current device is an sm_103 part (cached per device).
conv_status check_device();
// Time limit, in nanoseconds, of every wait inside a kernel.
uint64_t wait_limit_ns();
// Number of SMs of the current device.
int device_sm_count();
// Device address of the current device's status word (kernels record
// CONV_ERR_DEVICE_TIMEOUT there); nullptr if it cannot be obtained.
int *device_status_word();

}  // namespace i8c
