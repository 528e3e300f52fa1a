/*
 * int8conv.h -- C ABI of the GB300 (sm_103a) INT8 2-D convolution forward
 * propagation library, libint8conv.so.
 *
 * The operation is conv_fprop as defined in the cuDNN documentation page
 * "Convolutions", section "Convolution Fprop" (response = image * filter),
 * with the arguments of its "Python API" list: image, weight, pre_padding,
 * post_padding, stride, dilation, convolution_mode, compute_data_type; the
 * "symmetric-padding overload" (padding in place of pre/post) is
 * conv_params_set_symmetric_padding below.  Tensors are described as in the
 * forum thread "INT8 convolution using cuDNN Python Frontend": logical dims
 * plus one element stride per logical dim.
 *
 * Semantics (integer arithmetic throughout, exact):
 *   Y[n,k,p,q] = sum_{c,r,s} X[n,c,h,w] * W[k,c,r',s']   (+ bias[k]) (ReLU)
 *     h = p*stride[0] - pre_padding[0] + r*dilation[0]
 *     w = q*stride[1] - pre_padding[1] + s*dilation[1]
 *     taps outside the image contribute 0 (zero padding)
 *     (r',s') = (r,s) for CONV_CROSS_CORRELATION,
 *               (R-1-r, S-1-s) for CONV_CONVOLUTION (the filter flipped in
 *               both spatial axes; channels are not flipped)
 *     P = floor((H + pre[0] + post[0] - dilation[0]*(R-1) - 1) / stride[0]) + 1
 *     Q likewise with index 1.
 *   The accumulator is exact: the validator rejects shapes for which
 *   C*R*S*2^14 could exceed 2^31-1.  The bias is added with two's-complement
 *   int32 wrap-around, then ReLU is max(0, .).
 *
 * Ownership: the caller owns every buffer and the stream.  conv_fprop never
 * allocates and never synchronises; all work is queued on `stream`.  The
 * library keeps one small device status word per device (see
 * conv_device_status) and, in static host memory, the plan caches described
 * at conv_shutdown.
 *
 * Errors: every entry point returns a conv_status; nothing is thrown across
 * the ABI.  Descriptors are validated before anything is launched (a call
 * whose descriptors and parameters equal those of an earlier, validated call
 * reuses that validation from the plan cache).  Kernel launch failures give
 * CONV_ERR_CUDA.  A kernel whose internal wait runs out of time records
 * CONV_ERR_DEVICE_TIMEOUT in the
 * device status word and returns early; conv_device_status reports it.
 *
 * Thread safety: all entry points are reentrant; concurrent calls on
 * different streams are independent (they share only the status word).
 */
#ifndef INT8CONV_H
#define INT8CONV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV_OK = 0,
    CONV_ERR_NULL_PTR = 1,            /* a required pointer is NULL */
    CONV_ERR_RANK = 2,                /* a descriptor's rank is not 4 */
    CONV_ERR_DTYPE = 3,               /* image/filter not INT8; output not INT32 (INT8 with CONV_EPILOGUE_INT8_OUT) */
    CONV_ERR_SHAPE_MISMATCH = 4,      /* C, K, N or the output dims disagree */
    CONV_ERR_BAD_STRIDES = 5,         /* non-positive stride of a dim > 1, or elements alias */
    CONV_ERR_BUFFER_TOO_SMALL = 6,    /* descriptor's capacity_bytes below its extent */
    CONV_ERR_BAD_PARAM = 7,           /* stride/dilation < 1, padding < 0, empty output, bad mode */
    CONV_ERR_OVERFLOW_RISK = 8,       /* C*R*S*2^14 > 2^31-1: int32 could overflow */
    CONV_ERR_UNSUPPORTED_COMPUTE = 9, /* compute_dtype other than CONV_INT32 */
    CONV_ERR_ALIGNMENT = 10,          /* a forced algorithm cannot take these pointers/strides */
    CONV_ERR_CUDA = 11,               /* a CUDA runtime call failed */
    CONV_ERR_DEVICE_TIMEOUT = 12,     /* a kernel gave up waiting (see conv_device_status) */
    CONV_ERR_WORKSPACE = 13,          /* workspace NULL or smaller than conv_fprop_workspace_size */
    CONV_ERR_UNSUPPORTED_DEVICE = 14, /* the current device is not sm_103 */
    CONV_ERR_OVERLAP = 15,            /* output bytes overlap an input or the workspace */
    CONV_ERR_TOO_LARGE = 16,          /* an extent or offset exceeds the library's index range */
    CONV_ERR_STATIC_WORKSPACE_LIMIT = 17 /* call needs more scratch than CONV_STATIC_WORKSPACE_BYTES */
} conv_status;

typedef enum { CONV_INT8 = 1, CONV_INT32 = 2 } conv_dtype;

typedef enum { CONV_CROSS_CORRELATION = 0, CONV_CONVOLUTION = 1 } conv_mode;

/* Algorithm selection; CONV_ALGO_AUTO lets the planner choose. */
typedef enum {
    CONV_ALGO_AUTO = 0,
    CONV_ALGO_IMPLICIT_GEMM = 1, /* tcgen05 tensor-core implicit GEMM */
    CONV_ALGO_DIRECT_DP4A = 2,   /* CUDA-core direct kernel, 4-way int8 dot products */
    CONV_ALGO_DIRECT_GENERIC = 3, /* CUDA-core direct kernel, any strides */
    /* the tensor-core kernel with the image gathered by per-thread global
       loads instead of TMA im2col tiles (what CONV_ALGO_IMPLICIT_GEMM falls
       back to when a TMA im2col map cannot express the call: stride > 8,
       padding or reach beyond the map's corner range) */
    CONV_ALGO_IMPLICIT_GEMM_GLOBAL_LOADS = 4
} conv_algo;

/* Epilogue flags (bit set). */
#define CONV_EPILOGUE_BIAS 1u /* add int32 bias[k] */
#define CONV_EPILOGUE_RELU 2u /* max(0, .) after the bias */
/* int8 output: after bias and ReLU, v -> floor((v + 2^(s-1)) / 2^s) for
 * s = out_shift > 0 (a rounding right shift; s = 0 leaves v), then clamped to
 * [-128, 127].  The output descriptor must then be CONV_INT8 (and must be
 * CONV_INT32 without this flag: an output type is never inferred). */
#define CONV_EPILOGUE_INT8_OUT 4u

/*
 * Tensor descriptor.  dims and strides are in LOGICAL order: [N,C,H,W] for
 * the image and output ([N,K,P,Q]), [K,C,R,S] for the filter.  strides are in
 * elements (not bytes), one per logical dim, as in the forum thread's
 * graph.tensor(dim=..., stride=...).  The stride of a dim of extent 1 is
 * never multiplied by a non-zero index and is ignored.  capacity_bytes is the
 * size of the buffer behind the pointer; the largest addressed element must
 * lie inside it.
 */
typedef struct {
    int32_t dtype;          /* conv_dtype */
    int32_t rank;           /* must be 4 */
    int64_t dims[4];
    int64_t strides[4];
    uint64_t capacity_bytes;
} conv_tensor_desc;

/* conv_fprop attributes (cuDNN "Convolutions": Conv_fprop_attributes setters
 * and the Python argument list).  Index 0 is the H axis, index 1 the W axis. */
typedef struct {
    int64_t pre_padding[2];
    int64_t post_padding[2];
    int64_t stride[2];
    int64_t dilation[2];
    int32_t mode;          /* conv_mode */
    int32_t compute_dtype; /* must be CONV_INT32 */
    uint32_t epilogue;     /* CONV_EPILOGUE_* bits */
    int32_t algo;          /* conv_algo */
    int32_t out_shift;     /* 0..31, with CONV_EPILOGUE_INT8_OUT only (else 0) */
    int32_t reserved;      /* must be 0 */
} conv_fprop_params;

/* Fill *p with: no padding, stride 1, dilation 1, cross-correlation,
 * compute INT32, no epilogue, automatic algorithm, shift 0. */
void conv_params_init(conv_fprop_params *p);

/* The symmetric-padding overload: pre_padding = post_padding = pad. */
void conv_params_set_symmetric_padding(conv_fprop_params *p, const int64_t pad[2]);

/* Stride calculator: fill d for a packed tensor.  layout is one of "NCHW",
 * "NHWC" (image/output) or "KCRS", "KRSC" (filter); dims are logical.
 * capacity_bytes is set to the packed size.  Returns CONV_ERR_BAD_PARAM for
 * an unknown layout or a non-positive dim. */
conv_status conv_tensor_desc_packed(conv_tensor_desc *d, int32_t dtype, const int64_t dims[4],
                                    const char *layout);

/* Output dims [N,K,P,Q] for image x, filter w and params p. */
conv_status conv_fprop_output_dims(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                   const conv_fprop_params *p, int64_t out_dims[4]);

/* Full host-side validation of a call (no device work).  bias_elems is the
 * number of int32 elements behind the bias pointer (ignored unless the bias
 * flag is set; must be >= K when it is). */
conv_status conv_fprop_validate(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                const conv_tensor_desc *y, const conv_fprop_params *p,
                                int64_t bias_elems);

/* Algorithm the planner would run for this call (after validation). */
conv_status conv_fprop_plan(const conv_tensor_desc *x, const conv_tensor_desc *w,
                            const conv_tensor_desc *y, const conv_fprop_params *p,
                            int32_t *algo_out);

/* Bytes of device workspace conv_fprop needs for this call (0 for the direct
 * kernels; for the implicit GEMM the repacked half-precision filter, plus
 * the int32 partial sums of tiles whose reduction is cut over several SMs
 * (calls with fewer tiles than SMs and long reductions, or a short partial
 * last round of tiles), plus a channels-last copy of the image when its
 * strides allow neither direct channels-last loads nor whole-row loads: an
 * NCHW-like image, each channel's rows contiguous, is read in place when its
 * rows are at most 192 bytes (a multiple of 16), the stride along W is 1 and
 * Q, the pre-padding along W and every tap offset s*dilation_w are multiples
 * of 4, for K <= 192).  The caller allocates it, 256-byte
 * aligned.  The size assumes a
 * 16-byte-aligned image pointer (as every cudaMalloc or PyTorch allocation
 * is); with a misaligned one the image needs the copy too, and conv_fprop
 * returns CONV_ERR_WORKSPACE if the workspace cannot hold it. */
conv_status conv_fprop_workspace_size(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                      const conv_tensor_desc *y, const conv_fprop_params *p,
                                      size_t *bytes);

/* Number of kernels conv_fprop launches for this call, under the same
 * assumption of 16-byte aligned image and filter pointers: 0 for an empty
 * output, 1 for the direct kernels; for the implicit GEMM the filter repack
 * (none when the 128- or 192-column kernel converts the filter itself: K <=
 * 192, a channels-last (or copied) image, a filter with contiguous channels
 * and 16-byte aligned strides), the channels-last image copy when needed,
 * the convolution, and the reduction of cut tiles when the call cuts them.
 * (conv_fprop_pack_filter launches the repack, conv_fprop_prepacked the
 * others, the convolution then reading the repacked filter.)
 * Errors as conv_fprop_validate; CONV_ERR_NULL_PTR if count is NULL. */
conv_status conv_fprop_kernel_count(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                    const conv_tensor_desc *y, const conv_fprop_params *p, int32_t *count);

/* Tile shape of the implicit-GEMM convolution for this call, under the same
 * alignment assumption: shape[0] output pixels per tile (128), shape[1]
 * output channels per tile (128, 192 or 256: the smallest that covers K),
 * shape[2] the number of tiles, shape[3] the number of work units (whole
 * tiles, plus the runs of the tiles cut along the reduction: calls with
 * fewer tiles than SMs and long reductions, or a short partial last round,
 * on the current device).  All four are 0 for the direct kernels and for
 * an empty output.  Errors as conv_fprop_validate; CONV_ERR_NULL_PTR if
 * shape is NULL.  Host-only; no device work. */
conv_status conv_fprop_tile_shape(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                  const conv_tensor_desc *y, const conv_fprop_params *p, int64_t shape[4]);

/*
 * Y = conv_fprop(X, W) on `stream` (a cudaStream_t; NULL = legacy default).
 * x_dev, w_dev, y_dev, bias_dev and workspace are device pointers on the
 * current device.  bias_dev holds K int32 values and is read only when
 * p->epilogue has CONV_EPILOGUE_BIAS.  y_dev holds int32 elements, or int8
 * elements with CONV_EPILOGUE_INT8_OUT (as its descriptor says).  The output
 * must not overlap the inputs or the workspace.  Asynchronous: returns after
 * queuing the kernels.
 */
conv_status conv_fprop(const conv_tensor_desc *x, const int8_t *x_dev,
                       const conv_tensor_desc *w, const int8_t *w_dev,
                       const conv_tensor_desc *y, void *y_dev,
                       const int32_t *bias_dev, const conv_fprop_params *p,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * conv_fprop in two halves, for callers that reuse one filter across many
 * images (the filter repack then runs once):
 *   conv_fprop_pack_filter writes the repacked filter into the workspace
 *   (nothing to do for the direct kernels);
 *   conv_fprop_prepacked runs the convolution from that workspace.
 * Both take the same descriptors and params as conv_fprop and validate them
 * the same way; conv_fprop_prepacked still needs w_dev (the direct kernels
 * read the filter itself), and its tensor-core kernels always read the
 * repacked filter, also where conv_fprop would have them convert the filter
 * themselves.  The workspace contents must come from a
 * conv_fprop_pack_filter call with the same filter, descriptors and params;
 * the library cannot check that.  Calling the two in order on one stream is
 * conv_fprop.
 */
conv_status conv_fprop_pack_filter(const conv_tensor_desc *x, const conv_tensor_desc *w, const int8_t *w_dev,
                                   const conv_tensor_desc *y, const conv_fprop_params *p, void *workspace,
                                   size_t workspace_bytes, void *stream);

conv_status conv_fprop_prepacked(const conv_tensor_desc *x, const int8_t *x_dev,
                                 const conv_tensor_desc *w, const int8_t *w_dev,
                                 const conv_tensor_desc *y, void *y_dev,
                                 const int32_t *bias_dev, const conv_fprop_params *p,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * conv_fprop with the image, filter, bias and output in HOST memory (same
 * descriptors and semantics as conv_fprop; x_host, w_host, y_host and
 * bias_host are host pointers, page-locked for the copies to overlap).
 *
 * The filter and bias are copied once; the batch is then processed in a
 * short lead chunk (a quarter of a chunk, so that the copy back to the host
 * starts early) and up to four chunks of whole images on three
 * library-owned streams, so that the
 * copy of chunk c to the device, the convolution of chunk c-1 and the copy
 * of chunk c-2 back to the host run at the same time.  Chunking needs every
 * image in its own byte range of the buffers (batch outermost in memory, as
 * in NCHW or NHWC); otherwise the whole batch is one chunk.
 *
 * device_buffer (device memory, 256-byte aligned, at least
 * conv_fprop_host_buffer_size bytes, owned by the caller) holds the filter,
 * bias, workspace and double-buffered image and output chunks.  The call is
 * asynchronous: it returns after queueing the work, and `stream` (the
 * caller's) is made to wait for its completion, so synchronising `stream`
 * means y_host holds the result.  The streams and events it uses are created
 * on the first call on each device and live until the process exits; calls
 * on one device are queued one after the other.
 */
conv_status conv_fprop_host_buffer_size(const conv_tensor_desc *x, const conv_tensor_desc *w,
                                        const conv_tensor_desc *y, const conv_fprop_params *p,
                                        size_t *bytes);

conv_status conv_fprop_host(const conv_tensor_desc *x, const int8_t *x_host,
                            const conv_tensor_desc *w, const int8_t *w_host,
                            const conv_tensor_desc *y, void *y_host,
                            const int32_t *bias_host, const conv_fprop_params *p,
                            void *device_buffer, size_t device_buffer_bytes, void *stream);

/*
 * conv_fprop without a caller-provided workspace.  (The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory: a plugin whose host framework owns all device
 * allocations and hands none to it, or a latency-critical loop that must not
 * call cudaMalloc, which may synchronise the device.)
 *
 * Same arguments and results as conv_fprop, minus the workspace: the scratch
 * (the repacked filter; the int32 partial sums of the tiles whose reduction
 * a call cuts into runs for different SMs, which on a 32 x 256 x 56 x 56
 * 3x3 call are 18.9 MB of the 20.1 MB it needs; and, when the image strides
 * need it, a channels-last image copy) lives in a device array of
 * CONV_STATIC_WORKSPACE_BYTES that is part of the library, so every GPU that
 * loads the library holds that much memory until the process exits.  Calls needing more scratch than that
 * return CONV_ERR_STATIC_WORKSPACE_LIMIT and launch nothing
 * (conv_fprop_workspace_size tells the need in advance).  It allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 * The first call on a device looks up that device's copy of the array (one
 * cudaGetSymbolAddress with the device current), so make that first call
 * before any stream capture.  The address is kept per device ordinal for
 * the life of the device's primary context (the runtime's context): after
 * cudaDeviceReset, or with another context made current on that ordinal, it
 * is stale; use conv_fprop with a workspace there.  Every call shares the one array and the
 * kernels overwrite all scratch they read, so nothing needs clearing between
 * calls; but calls whose work overlaps on the GPU (different streams, or
 * different host threads) race on the array: order them on one stream.
 */
#define CONV_STATIC_WORKSPACE_BYTES (32u << 20)

conv_status conv_fprop_static_workspace(const conv_tensor_desc *x, const int8_t *x_dev,
                                        const conv_tensor_desc *w, const int8_t *w_dev,
                                        const conv_tensor_desc *y, void *y_dev,
                                        const int32_t *bias_dev, const conv_fprop_params *p,
                                        void *stream);

/*
 * Gradients of the same convolution (cuDNN "Convolutions", sections
 * "Convolution Dgrad" and "Convolution Wgrad": the data and weight gradients
 * during backpropagation).  The pages name the operations and their
 * arguments but print no formula; they are computed as the transposes of
 * the forward sum:
 *
 *   dX[n,c,h,w]   = sum over k, r, s of dY[n,k,p,q] * W[k,c,r',s'],
 *                   p = (h + pre_h - r*dil_h) / stride_h when that division
 *                   is exact and 0 <= p < P (q likewise),
 *   dW[k,c,r',s'] = sum over n, p, q of dY[n,k,p,q] * X[n,c,h,w],
 *                   h = p*stride_h - pre_h + r*dil_h (w likewise), zero
 *                   outside the image,
 *
 * with (r', s') = (r, s) in CROSS_CORRELATION and (R-1-r, S-1-s) in
 * CONVOLUTION, exactly as conv_fprop pairs image and filter elements.
 *
 * Descriptors: dy is the loss gradient, int8 [N,K,P,Q]; w and x as in
 * conv_fprop (int8); dx is int32 [N,C,H,W] and dw int32 [K,C,R,S], any
 * strides.  H, W (dgrad) and R, S (wgrad) come from the output descriptor;
 * P, Q must be the forward output size for them.  p is the forward call's
 * parameters with no epilogue (epilogue and out_shift 0) and algo AUTO,
 * IMPLICIT_GEMM or DIRECT_GENERIC.  Results are exact: dgrad needs
 * K*R*S*2^14 <= 2^31-1 and wgrad N*P*Q*2^14 <= 2^31-1, else
 * CONV_ERR_OVERFLOW_RISK.
 *
 * conv_dgrad runs on the tensor cores as stride_h*stride_w forward
 * convolutions of dY, one per residue class (h mod stride_h, w mod
 * stride_w) of dX's pixels, each by the filter taps that reach that class
 * (taken backwards, K and C exchanged) with stride 1, each in its own part of
 * the workspace; the filters of all classes are repacked by one launch on
 * `stream`, a dY that is neither channels-last nor read in place by rows
 * (as for conv_fprop's image) is copied once for all classes,
 * and the classes run as one kernel launch on `stream` (each on its share
 * of the SMs) when they use the same kernel variant and cut no tiles;
 * otherwise side by side on up to four library-owned streams forked from
 * `stream` and joined back to it (events; streams and events are created on
 * the first such call on a device, so make that call outside a stream
 * capture; one such call at a time per device forks and joins, the others
 * wait on a host mutex); a class no tap reaches is written with zeros.
 * More than 64 classes take the CUDA-core kernel.  conv_wgrad runs on the
 * tensor cores as a forward convolution of the image (batch and channel
 * dims exchanged) by dY (its batch as channels, its pixels as taps) when the
 * tensor-core kernel can express it; with a batch of at most 32 it folds T
 * = min(64 / N, Q, 8) columns of dY into the channels, reading a copy of
 * the image T times its size.  Those routes need the workspace the
 * *_workspace_size call reports (256-byte aligned, caller-owned; for dgrad
 * it holds every class's filter repacked to f16 blocks, for wgrad dY
 * repacked to f16 blocks, about 2*K*P*ceil(Q/T)*64 bytes (T = 1 unfolded,
 * times ceil(N/64)), plus the int32 partial sums of the reduction split over
 * the SMs, plus the folded image copy, C*H*U*ceil(T*N/16)*16 bytes with U
 * about T*stride_w*ceil(Q/T) + dilation_w*(S-1)).  Other calls, and algo
 * DIRECT_GENERIC, run CUDA-core kernels and need none; IMPLICIT_GEMM on a
 * call that cannot take the tensor cores returns CONV_ERR_ALIGNMENT.
 * Pointers are device pointers on the current device, outputs must not
 * overlap inputs or the workspace; the calls are asynchronous on `stream`
 * and allocate nothing.  An empty dX (N, C, H or W zero) is a no-op; an
 * empty batch in conv_wgrad writes an all-zero dW and reads neither input,
 * so x_dev and dy_dev may then be null.
 */
conv_status conv_dgrad_workspace_size(const conv_tensor_desc *dy, const conv_tensor_desc *w,
                                      const conv_tensor_desc *dx, const conv_fprop_params *p, size_t *bytes);
conv_status conv_dgrad(const conv_tensor_desc *dy, const int8_t *dy_dev, const conv_tensor_desc *w,
                       const int8_t *w_dev, const conv_tensor_desc *dx, int32_t *dx_dev,
                       const conv_fprop_params *p, void *workspace, size_t workspace_bytes, void *stream);
conv_status conv_wgrad_workspace_size(const conv_tensor_desc *x, const conv_tensor_desc *dy,
                                      const conv_tensor_desc *dw, const conv_fprop_params *p, size_t *bytes);
conv_status conv_wgrad(const conv_tensor_desc *x, const int8_t *x_dev, const conv_tensor_desc *dy,
                       const int8_t *dy_dev, const conv_tensor_desc *dw, int32_t *dw_dev,
                       const conv_fprop_params *p, void *workspace, size_t workspace_bytes, void *stream);

/* Synchronise `stream`, then read and clear the current device's status
 * word: CONV_OK, or CONV_ERR_DEVICE_TIMEOUT if a kernel gave up waiting
 * since the last call. */
conv_status conv_device_status(void *stream);

/* Self-test of the timeout path: launches one kernel that waits on a barrier
 * nobody signals, with a limit of `limit_us` microseconds, so that it records
 * CONV_ERR_DEVICE_TIMEOUT and exits.  Returns the launch status. */
conv_status conv_selftest_wait_timeout(uint32_t limit_us, void *stream);

/*
 * Peak microbenchmark: the measured rates of the instruction routes an exact
 * int8 product can take on the current device, and its copy bandwidth.  The
 * pages quote no peak; the benchmark divides by these (or by the driver's
 * measured bf16 rate and copy bandwidth) instead of a datasheet figure.
 * sm_103a has no integer kind of tcgen05.mma, so the routes are:
 *   tcgen05_f16_tflops   tcgen05.mma.cta_group::1.kind::f16, M=128 N=256
 *                        K=16, f32 accumulators in tensor memory, one CTA
 *                        per SM issuing back to back (the route the
 *                        convolution kernel takes, exact by grouping);
 *   mma_sync_s8_tops     warp-level mma.sync m16n8k32 s8 x s8 -> s32;
 *   mma_sync_f16_tflops  warp-level mma.sync m16n8k16 f16 x f16 -> f32;
 *   dp4a_tops            the CUDA cores' dp4a (4 products + 4 adds);
 *   hbm_copy_gbs         read + write bytes per second of a 16-byte copy
 *                        kernel over the two halves of `scratch` (0 when
 *                        scratch_bytes is below 512 MiB + 4 KiB);
 *   sm_mhz               SM clock during the tcgen05 run (clock64 cycles per
 *                        global-timer nanosecond).
 * Rates count 2 operations per multiply-add, dense.  Each kernel runs about
 * a millisecond (best of three launches timed with events on `stream`).
 * `scratch`: caller-owned device buffer, 256-byte aligned, at least 1 MiB
 * (timing records; the copy uses the rest).  Synchronises `stream`; not
 * for use inside a stream capture.  Errors: CONV_ERR_NULL_PTR,
 * CONV_ERR_WORKSPACE (scratch too small or misaligned), CONV_ERR_CUDA,
 * CONV_ERR_DEVICE_TIMEOUT (an MMA completion wait ran out).
 */
typedef struct {
    double tcgen05_f16_tflops;
    double mma_sync_s8_tops;
    double mma_sync_f16_tflops;
    double dp4a_tops;
    double hbm_copy_gbs;
    double sm_mhz;
} conv_peak_rates;

conv_status conv_measure_peak_rates(void *scratch, size_t scratch_bytes, conv_peak_rates *out, void *stream);

/*
 * Plan caches (the cuDNN-frontend tutorial's kernel/plan cache, for repeated
 * calls of one shape): conv_fprop, its two halves, the static-workspace and
 * host-buffer variants and the gradients' forward convolutions keep
 *   - the validated geometry, algorithm and tensor-core plan of a call,
 *     keyed by the three descriptors, the parameters, the device and whether
 *     the image pointer is 16-byte aligned (64 entries), and
 *   - the tensor-core kernel's launch arguments with their encoded TMA
 *     tensor maps, keyed by that plan and the 16-byte alignment of the image
 *     and output pointers (32 entries); a call with other buffers re-targets
 *     the cached maps to its addresses (cuTensorMapReplaceAddress) instead of
 *     encoding them again;
 *   - for conv_dgrad, the residue classes with their tensor-core plans,
 *     keyed like the first cache on dY, W, dX and the parameters (16
 *     entries).
 * A call whose key is cached skips validation, planning and map encoding;
 * its pointer checks (null, overlap, workspace) still run.  The caches are
 * library-owned host memory, shared by all threads (a mutex guards them),
 * least recently used entries giving way.  Cache lookups make no CUDA calls,
 * so cached calls stay capturable in CUDA graphs.
 *
 * conv_shutdown empties the three caches (their memory is static; nothing is
 * freed or allocated; the data gradient's side streams and events stay).  Call it when no other thread is inside a library
 * call.  conv_plan_cache_stats reads the hit and miss counts since the
 * library was loaded.
 */
void conv_shutdown(void);
conv_status conv_plan_cache_stats(uint64_t *plan_hits, uint64_t *plan_misses, uint64_t *launch_hits,
                                  uint64_t *launch_misses);

/* Human-readable name of a status. */
const char *conv_status_string(conv_status s);

/* Library version, major*10000 + minor*100 + patch. */
int32_t conv_library_version(void);

#ifdef __cplusplus
}
#endif

#endif /* INT8CONV_H */
