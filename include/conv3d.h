/*
 * conv3d.h -- C ABI of libconv3d.so: forward implicit-GEMM convolution
 * (conv3d; conv2d and conv1d as the degenerate D=T=1 / H=R=1 forms) over
 * channel-last NDHWC activations and KTRSC weights on one GB300 (sm_103a),
 * plus the NCDHW -> NDHWC layout / fp8-e4m3 quantisation pack.
 *
 * Where each operation is defined (pages of the method):
 *   - conv_fwd: FlyDSL PR #860 "fp8 conv3d: 8-wave GEMM pipeline + BIG_IN
 *     fix" -- PR summary (the conv as a GEMM: M = output positions, N = K
 *     filters, reduction over crs = C*T*R*S; weight = a plain KTRSC (k, crs)
 *     matrix; E4M3FN fp8 inputs; fp32 accumulation), and its commits on the
 *     temporal-only 3x1x1 decode, >2^31-element addressing, split-K and the
 *     conv2d/conv1d reshape wrappers.  Point-output (patch-embedding) shapes
 *     are one plain GEMM: MIOpen PR #10912 "Use a single GEMM for
 *     point-output conv in all three directions", description.
 *   - conv_fwd_ncdhw: the same conv reading a channel-major activation in
 *     place, the NCDHW-direct kernel FlyDSL PR #860's 3x1x1 / 1x1x1 commits
 *     leave to future work.
 *   - pack_ncdhw_bf16_to_ndhwc(_fp8): FlyDSL PR #860, commit adding the
 *     tiled NCDHW->NDHWC bf16->fp8 pack kernel (replacing torch.permute) and
 *     the commit fixing its >2 GB addressing.
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense and contiguous, in the stated layout.  Every
 *     device pointer must be 16-byte aligned.
 *   - The caller owns and allocates every buffer (inputs, outputs, scales,
 *     workspace).  The library never allocates or frees caller memory.  It
 *     keeps only a per-device status word, per-process host state
 *     (function pointers, device attributes) and, once conv_fwd_from_host
 *     has run on a device, two copy streams and a set of events there.
 *     That per-device state lives until the process exits: after
 *     cudaDeviceReset on a device, do not use the library on that device
 *     again in the same process.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and do
 *     not synchronise the host, except conv_get_device_status(_stream).
 *   - Every function returns a conv_status; no exception crosses the ABI.
 *     On any non-OK return nothing has been launched (conv_fwd_from_host:
 *     see there).
 *   - Shapes are int64; tensors above 2^31 elements (and 2^32 bytes) are
 *     supported; each single dimension must be below 2^31.
 */
#ifndef CONV3D_GB300_H
#define CONV3D_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV_OK = 0,
    CONV_ERR_INVALID = 1,     /* null pointer, bad dims, C mismatch, misaligned pointer */
    CONV_ERR_UNSUPPORTED = 2, /* shape the kernels do not cover (see conv_fwd) */
    CONV_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
    CONV_ERR_TIMEOUT = 4      /* a kernel gave up on a bounded wait (device status) */
} conv_status;

typedef enum {
    CONV_DTYPE_BF16 = 0,      /* x, w: bfloat16 */
    CONV_DTYPE_FP8_E4M3 = 1   /* x, w: fp8 E4M3FN bytes, dequantised by scale_x / scale_w */
} conv_dtype;

/* Dispatch classes chosen by conv_fwd (reported by conv_fwd_plan). */
typedef enum {
    CONV_CLASS_GENERIC = 0,   /* implicit GEMM, A gathered by TMA im2col */
    CONV_CLASS_TEMPORAL = 1,  /* T x 1 x 1 filter, unit H/W stride, no H/W pad: tiled TMA rows */
    CONV_CLASS_POINT_GEMM = 2,/* point-output / pointwise conv: one plain GEMM */
    CONV_CLASS_PATCH_GEMM = 3,/* stride == filter patches the implicit classes cannot read:
                                 gathered into GEMM rows in the workspace, then one GEMM */
    CONV_CLASS_NONE = -1
} conv_class;

/* Output dims of the forward conv (torch semantics: floor((in + 2p - d(f-1) - 1)/s) + 1).
 *   x_dims  = {N, D, H, W, C}     activation, NDHWC
 *   w_dims  = {K, T, R, S, C}     weight, KTRSC
 *   stride, pad, dil = {d, h, w}  pad is symmetric per dimension
 *   out_dims (out) = {N, Do, Ho, Wo, K}
 * Returns CONV_ERR_INVALID for non-positive dims/strides/dilations, negative
 * pads, C mismatch, or an empty output.  Host-only; needs no GPU. */
int conv_out_dims(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                  const int pad[3], const int dil[3], int64_t out_dims[5]);

/* The plan conv_fwd would run for this problem on the current device
 * (class, tile N, bytes per k-step row, pipeline stages, split-K factor,
 * CTAs launched), and the workspace bytes it needs for split-K.  Any output
 * pointer may be NULL.  If no workspace (or a smaller one) is given to
 * conv_fwd, it runs the same plan without split-K.  num_sms <= 0 means "ask
 * the current device" (needs a GPU); a positive value plans for that many
 * SMs host-only.  Returns CONV_ERR_UNSUPPORTED when conv_fwd would. */
int conv_fwd_plan(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                  const int pad[3], const int dil[3], int dtype, int num_sms, int* cls,
                  int* tile_n, int* k_bytes, int* stages, int* splits, int* ctas,
                  size_t* workspace_bytes);

/* Bytes of device workspace conv_fwd uses for this problem on the current
 * device: the workspace_bytes conv_fwd_plan reports (split-K partials,
 * aligned operand copies of a point-output GEMM, the gathered rows of the
 * patch class).  0 when the plan needs none, and also when the problem is
 * invalid or unsupported or no GPU is usable (conv_fwd_plan returns the
 * status, conv_last_error describes it).  Needs a GPU.  The split-K rule it
 * sizes follows FlyDSL PR #860's split-K commits (split the reduction when
 * the output tiles leave the GPU under-filled). */
size_t conv_fwd_workspace_size(const int64_t x_dims[5], const int64_t w_dims[5],
                               const int stride[3], const int pad[3], const int dil[3],
                               int dtype);

/* Number of kernels conv_fwd launches for this problem and workspace size on
 * the current device (operand copies / patch gather, the convolution's
 * launches -- long reductions run as several launches of whole waves --, and
 * the split-K reduction).  Needs a GPU. */
int conv_fwd_kernel_launches(const int64_t x_dims[5], const int64_t w_dims[5],
                             const int stride[3], const int pad[3], const int dil[3], int dtype,
                             size_t workspace_bytes, int* launches);

/* Forward convolution:
 *   out[n,od,oh,ow,k] = bf16_rn( scale_x * scale_w *
 *       sum_{t,r,s,c} x[n, od*sd-pd+t*dd, oh*sh-ph+r*dh, ow*sw-pw+s*dw, c] * w[k,t,r,s,c] )
 * with x = 0 outside the input (zero padding; cross-correlation, no flip),
 * products of the exact bf16 / e4m3 input values accumulated in fp32.
 *   x        device, NDHWC [N,D,H,W,C], bf16 or e4m3 per dtype
 *   w        device, KTRSC [K,T,R,S,C], same dtype as x
 *   scale_x, scale_w  device pointers to one fp32 each, or NULL for 1.0
 *   out      device, NDHWC [N,Do,Ho,Wo,K] bf16; fully overwritten
 *   workspace, workspace_bytes  device scratch for split-K partials (may be
 *            NULL/0: split-K is then not used); size from conv_fwd_plan
 * Coverage: C*elem_bytes % 16 == 0 for the implicit-GEMM classes; the
 * point-output class needs T*R*S*C*elem_bytes % 4 == 0; strides <= 8 and
 * pads <= 15 for the im2col class.  Convolutions with stride == filter and
 * zero padding outside those limits (e.g. 14x14 or 16x16 patches of an RGB
 * image) take the patch class, whose gathered rows need workspace
 * (conv_fwd_plan's size; a smaller one returns CONV_ERR_INVALID).  Anything
 * else: CONV_ERR_UNSUPPORTED (there is no fallback path).  Device-side wait
 * timeouts are reported by conv_get_device_status, not by this return value. */
int conv_fwd(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
             const int stride[3], const int pad[3], const int dil[3], int dtype,
             const float* scale_x, const float* scale_w, void* out, void* workspace,
             size_t workspace_bytes, cudaStream_t stream);

/* conv_fwd plus a per-filter bias:
 *   out[n,od,oh,ow,k] = bf16_rn( scale_x * scale_w * (the conv_fwd sum) + bias[k] )
 *   bias   device, fp32 [K], 4-byte aligned; NULL gives conv_fwd exactly
 * Every other argument, the plan and the error behaviour are conv_fwd's (with
 * split-K the bias is added once, in the reduction).  Defined by: FlyDSL PR
 * #860, PR summary, which lists bias among the fp8 conv's test cases; the
 * page gives neither the bias type nor where it enters, so it is taken as an
 * fp32 vector added after the dequantisation scales, before the rounding. */
int conv_fwd_bias(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
                  const int stride[3], const int pad[3], const int dil[3], int dtype,
                  const float* scale_x, const float* scale_w, const float* bias, void* out,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Epilogue activations of conv_fwd_bias_act. */
typedef enum {
    CONV_ACT_NONE = 0,
    CONV_ACT_RELU = 1,   /* max(v, 0) */
    CONV_ACT_SILU = 2,   /* v * sigmoid(v) = v / (1 + exp(-v)) */
    CONV_ACT_GELU = 3    /* v * Phi(v) = v/2 * (1 + erf(v / sqrt(2))), the erf form */
} conv_act;

/* conv_fwd_bias followed by an elementwise activation, applied in fp32 to
 * each output before the bf16 rounding:
 *   out[n,od,oh,ow,k] = bf16_rn( act( scale_x * scale_w * (the conv_fwd sum) + bias[k] ) )
 *   act    one of conv_act; anything else returns CONV_ERR_INVALID
 * GELU's erf is evaluated by Abramowitz & Stegun 7.1.26 (|error| <= 1.5e-7)
 * and the sigmoid with an approximate reciprocal, both far below the bf16
 * output's resolution.  Plans with an activation store through the direct
 * (non-staged) epilogue.  bias may be NULL.  Every other argument, the plan and the error behaviour
 * are conv_fwd_bias's (with split-K the activation is applied once, in the
 * reduction, after the bias).  Defined by: FlyDSL PR #860, PR summary, which
 * lists a bias case among the fp8 conv's tests; the pages name no activation
 * function, so the usual epilogue extension of that bias is offered in three
 * common forms, each as its textbook definition. */
int conv_fwd_bias_act(const void* x, const int64_t x_dims[5], const void* w,
                      const int64_t w_dims[5], const int stride[3], const int pad[3],
                      const int dil[3], int dtype, const float* scale_x, const float* scale_w,
                      const float* bias, int act, void* out, void* workspace,
                      size_t workspace_bytes, cudaStream_t stream);

/* conv_fwd_bias over a channel-major (NCDHW) activation, read in place: no
 * NCDHW -> NDHWC pass before the convolution.
 *   out[n,od,h,w,k] = bf16_rn( scale_x * scale_w *
 *       sum_{t,c} x[n, c, od*sd-pd+t*dd, h, w] * w[k,t,0,0,c] + bias[k] )
 *   x        device, NCDHW [N,C,D,H,W] bf16, 16-byte aligned
 *   x_dims   = {N, C, D, H, W}  (channel-major order, unlike conv_fwd)
 *   w        device, KTRSC [K,T,1,1,C] bf16
 *   out      device, NDHWC [N,Do,H,W,K] bf16 (conv_out_dims of the NDHWC
 *            view); fully overwritten
 *   stride, pad, dil, scale_x, scale_w, bias, workspace, stream: as for
 *            conv_fwd_bias (workspace size from conv_fwd_ncdhw_plan)
 * Coverage: bf16; T x 1 x 1 filters (any T, temporal stride, pad and
 * dilation; T = 1 is the pointwise conv) with unit H/W stride and no H/W
 * padding; H*W and C multiples of 8.  Anything else: CONV_ERR_UNSUPPORTED
 * (no fallback).  Each tap's A tile is 128 consecutive H*W positions of one
 * input plane by a block of channels, loaded as position-contiguous
 * (MN-major) TMA boxes.  Exception: with T > 1, C % 16 == 0, channel planes
 * (D*H*W*2 bytes) above 1 MiB and a workspace that holds an NDHWC copy of x
 * (the size conv_fwd_ncdhw_plan reports), x is first packed into that copy
 * and the copy convolved: in-place reads of such planes, revisited by every
 * tap, thrash address translation and L2 (three times the DRAM reads).  A
 * smaller workspace keeps the in-place reads; the result is the same.  Defined by: FlyDSL PR #860, the commits that drop
 * the 3x1x1 unfold path (a kernel reading NCDHW straight into the GEMM,
 * without materialising A, is left to future work) and the 1x1x1 matmul
 * path (the NCDHW -> NDHWC transpose costs about 5-6 ms of the 8.7 ms
 * pointwise conv); the math is conv_fwd's.  An fp8 variant that quantises
 * while loading is not covered. */
int conv_fwd_ncdhw(const void* x, const int64_t x_dims[5], const void* w, const int64_t w_dims[5],
                   const int stride[3], const int pad[3], const int dil[3], int dtype,
                   const float* scale_x, const float* scale_w, const float* bias, void* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* e4m3 forward convolution of a bf16 channel-major (NCDHW) activation, the
 * activation quantised while the kernel loads it -- no NCDHW -> NDHWC pack
 * pass and no packed copy:
 *   amax   = max |x| over the whole tensor (one read-only pass first)
 *   scale  = amax / 448 (1.0 if amax == 0), written to *scale_x_out
 *   q[n,c,d,h,w] = e4m3_satfinite_rn( fp32(x[n,c,d,h,w]) / scale )
 *   out[n,d,h,w,k] = bf16_rn( scale * scale_w *
 *       sum_{r,s,c} q[n, c, d, h+r-ph, w+s-pw] * w[k,0,r,s,c] + bias[k] )
 * so the result is conv_fwd_bias of pack_ncdhw_bf16_to_ndhwc_fp8(x) (the
 * same codes and scale) up to the fp32 summation order.
 *   x          device, bf16 NCDHW [N,C,D,H,W]; x_dims = {N, C, D, H, W}
 *   w          device, e4m3 KTRSC [K,1,R,S,C] (pack_ncdhw_bf16_to_ndhwc_fp8
 *              of the bf16 KCTRS weight, which also gives scale_w)
 *   scale_w    device fp32 or NULL (1.0); scale_x_out device fp32 or NULL
 *   bias       device fp32 [K] or NULL
 *   out        device, bf16 NDHWC [N,D,H,W,K]; fully overwritten
 *   workspace  device, >= pack_fp8_workspace_size() bytes (the amax word);
 *              with conv_fwd_ncdhw_fp8_workspace_size() bytes the converted
 *              strips are kept for the other column tiles (faster; same result)
 * Coverage: T = 1, odd R and S with pad = (0, (R-1)/2, (S-1)/2), unit
 * stride and dilation, C % 16 == 0; anything else CONV_ERR_UNSUPPORTED.
 * Each CTA converts, per 128-channel chunk, a strip of its output rows plus
 * the filter's reach into e4m3 in shared memory once; every tap reads the
 * strip in place, shifted.  A CTA (pair) computes all column tiles of an
 * m-tile in turn; with room in the workspace, the strips converted for the
 * first column tile are copied out (bulk copies, L2-resident) and copied
 * back for the others instead of being converted again.  Defined by: FlyDSL PR #860, the 3x1x1 unfold
 * revert commit (a kernel reading NCDHW straight into the GEMM, without
 * materialising A, left to future work) and the tiled bf16 -> fp8 pack
 * commit (the quantisation it folds in). */
int conv_fwd_ncdhw_fp8(const void* x, const int64_t x_dims[5], const void* w,
                       const int64_t w_dims[5], const int stride[3], const int pad[3],
                       const int dil[3], const float* scale_w, float* scale_x_out,
                       const float* bias, void* out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Preferred workspace bytes of conv_fwd_ncdhw_fp8 for this problem on the
 * current device (the amax word plus the kept strips: CTAs x 128-channel
 * chunks x strip bytes).  Returns CONV_ERR_UNSUPPORTED when the conv would. */
int conv_fwd_ncdhw_fp8_workspace_size(const int64_t x_dims[5], const int64_t w_dims[5],
                                      const int stride[3], const int pad[3], const int dil[3],
                                      size_t* bytes);

/* conv_fwd_plan for conv_fwd_ncdhw (x_dims = {N, C, D, H, W}); the class is
 * always CONV_CLASS_TEMPORAL.  Host-only when num_sms > 0. */
int conv_fwd_ncdhw_plan(const int64_t x_dims[5], const int64_t w_dims[5], const int stride[3],
                        const int pad[3], const int dil[3], int dtype, int num_sms, int* cls,
                        int* tile_n, int* k_bytes, int* stages, int* splits, int* ctas,
                        size_t* workspace_bytes);

/* conv_fwd with the operands and the result in HOST memory: the same
 * convolution (same definition and plan as conv_fwd, so the same output
 * bits), with the host->device copies of x and w and the device->host copy
 * of out overlapped with the convolution.
 *   x_host, w_host    host, NDHWC / KTRSC as for conv_fwd (page-locked for
 *                     the copies to overlap; pageable memory works, serially)
 *   out_host          host, NDHWC [N,Do,Ho,Wo,K] bf16; fully overwritten
 *   x_dev, w_dev, out_dev  device buffers of the same sizes (caller-owned,
 *                     16-byte aligned); on completion they hold copies of
 *                     x, w and out
 *   scale_x, scale_w  device pointers or NULL, as for conv_fwd
 *   workspace, workspace_bytes  as for conv_fwd
 *   chunks            0: automatic; 1: no overlap; n > 1: n slices (<= 32)
 * The output rows are cut into slices of whole waves of work units (with
 * chunks == 0: a first slice of one to four blocks of waves, chosen for the
 * fewest bytes ahead of its first launch, then one block, then slices
 * doubling up to a sixth of the rest, and one block last).  Before slice i
 * runs, the input rows it reads that are not on the device yet -- whole
 * (n, d) planes of x up to its last output plane's reach, and the leading H
 * rows of the planes that plane reaches -- are copied on a library-owned
 * copy-in stream; the kernel for slice i's output rows runs on `stream`
 * once they have landed, and slice i's output rows go back on a copy-out
 * stream while slice i+1 computes.  When the first slice spans several
 * waves over all column tiles, only the weight rows of its first group of
 * column tiles come before its first launch, and that slice runs as one
 * launch per group, each after its rows have landed.
 * Work queued on `stream` before the call runs before the copies; work
 * queued after it runs after the last copy: synchronise `stream` before
 * reading out_host.  Point-output GEMM and split-K plans run unsliced (copy
 * in, conv_fwd, copy out on `stream`).  The first call on a device creates
 * the two copy streams and the events with that device current.  Calls on
 * one device are enqueued one at a time (a lock); their copies share the
 * copy streams.  If an enqueue step fails after earlier steps were queued,
 * the call returns the error with `stream` still ordered after whatever was
 * queued.  The pages of the method have no counterpart: it is the measured
 * end-to-end path from host operands. */
int conv_fwd_from_host(const void* x_host, const int64_t x_dims[5], const void* w_host,
                       const int64_t w_dims[5], const int stride[3], const int pad[3],
                       const int dil[3], int dtype, const float* scale_x, const float* scale_w,
                       void* out_host, void* x_dev, void* w_dev, void* out_dev, void* workspace,
                       size_t workspace_bytes, int chunks, cudaStream_t stream);

/* The slices conv_fwd_from_host would cut this problem into (the same plan
 * and rule; a query: nothing is launched or copied).  num_sms > 0 plans for
 * that SM count without touching a device (232448 bytes of shared memory
 * per block), 0 for the current device; workspace_bytes and chunks as given
 * to conv_fwd_from_host (0: no workspace).  Writes *n_slices (1..32),
 * *weight_groups (the launches the first slice runs as, one per group of
 * column tiles), and for slice i:
 *   rows[2i], rows[2i+1]   its output rows [lo, hi) (row = (n, od, oh, ow));
 *   reach[3i .. 3i+2]      (whole, part, rows): the input on the device once
 *                          its copy-in has landed, as (n, d) planes of x,
 *                          planes [0, whole) entirely and rows [0, rows) of
 *                          planes [whole, part); the last slice: all of x.
 * rows holds 64 and reach 96 entries.  Returns CONV_ERR_INVALID for a null
 * pointer or chunks < 0, else as conv_fwd_plan. */
int conv_fwd_from_host_slices(const int64_t x_dims[5], const int64_t w_dims[5],
                              const int stride[3], const int pad[3], const int dil[3], int dtype,
                              int num_sms, size_t workspace_bytes, int chunks, int* n_slices,
                              int64_t* rows, int64_t* reach, int* weight_groups);

/* Backward passes of the point-output conv (MIOpen PR #10912 "Use a single
 * GEMM for point-output conv in all three directions": backward data and
 * backward weights of patch-embedding shapes, each one GEMM).  Shapes: zero
 * padding and x spatially equal to w's filter (D == T, H == R, W == S), so
 * the output is [N,1,1,1,K]; anything else returns CONV_ERR_UNSUPPORTED.
 * bf16 operands, fp32 accumulation, bf16 results; J = T*R*S*C.
 *   conv_bwd_data_point:   dx[n, j] = sum_k dy[n, k] * w[k, j]
 *       dy device [N,1,1,1,K]; w device KTRSC; dx device NDHWC (x's shape)
 *   conv_bwd_weight_point: dw[k, j] = sum_n dy[n, k] * x[n, j]
 *       x device NDHWC; dy device [N,1,1,1,K]; dw device KTRSC (w's shape)
 * x_dims / w_dims / stride / pad / dil describe the forward conv.  Both
 * transpose operands K-major into `workspace` (dx: w^T [J, K]; dw: x^T
 * [J, N'], N' = N rounded up to 8, zero-padded, and -- unless K % 8 == 0,
 * when dy is read in place as an MN-major operand -- dy^T [K, N']) and run
 * the pointwise forward GEMM on them (split-K over the batch for dw when the
 * rest of the workspace holds the partials).  A workspace smaller than the
 * transposes returns CONV_ERR_INVALID; conv_bwd_point_workspace_bytes
 * (which = 0 data, 1 weights) gives the preferred size.  Outputs are fully
 * overwritten; asynchronous on `stream`. */
int conv_bwd_point_workspace_bytes(const int64_t x_dims[5], const int64_t w_dims[5],
                                   const int stride[3], const int pad[3], const int dil[3],
                                   int which, size_t* bytes);
int conv_bwd_data_point(const void* dy, const void* w, const int64_t x_dims[5],
                        const int64_t w_dims[5], const int stride[3], const int pad[3],
                        const int dil[3], void* dx, void* workspace, size_t workspace_bytes,
                        cudaStream_t stream);
int conv_bwd_weight_point(const void* x, const void* dy, const int64_t x_dims[5],
                          const int64_t w_dims[5], const int stride[3], const int pad[3],
                          const int dil[3], void* dw, void* workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/* Layout pack: out[n,d,h,w,c] = in[n,c,d,h,w] (bit copy).
 *   in   device, bf16 NCDHW, dims = {N, C, D, H, W}
 *   out  device, bf16 NDHWC [N,D,H,W,C]
 * Also the weight pack: a torch weight [K,C,T,R,S] passed as N=K, D=T,
 * H=R, W=S gives the KTRSC weight conv_fwd takes. */
int pack_ncdhw_bf16_to_ndhwc(const void* in, const int64_t dims[5], void* out,
                             cudaStream_t stream);

/* Bytes of device workspace pack_ncdhw_bf16_to_ndhwc_fp8 needs (16). */
size_t pack_fp8_workspace_size(void);

/* Layout pack with per-tensor fp8 quantisation:
 *   amax  = max |in| over the whole tensor
 *   scale = amax / 448 (fp32, IEEE round to nearest; 1.0 if amax == 0)
 *   out[n,d,h,w,c] = e4m3_satfinite_rn( fp32(in[n,c,d,h,w]) / scale )
 *   in         device, bf16 NCDHW, dims = {N, C, D, H, W}
 *   out        device, e4m3 NDHWC
 *   scale_out  device, one fp32: receives scale (the dequantisation
 *              multiplier to pass to conv_fwd as scale_x or scale_w)
 *   workspace  device, >= pack_fp8_workspace_size() bytes of scratch
 * Non-finite inputs are not supported. */
int pack_ncdhw_bf16_to_ndhwc_fp8(const void* in, const int64_t dims[5], void* out,
                                 float* scale_out, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* Size of the static device scratch conv_fwd_noalloc uses: 8 MiB. */
#define CONV_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* conv_fwd for callers that cannot allocate device memory.  The pages of the
 * method have no counterpart of this entry point.
 *
 * conv_fwd takes its split-K scratch from the caller.  Some callers cannot
 * provide one: code that must not call cudaMalloc at run time (engines that
 * reserve all device memory up front, or latency-bound code that cannot
 * afford cudaMalloc's implicit device synchronisation).  This entry point
 * takes the same arguments as conv_fwd minus the workspace, runs the same
 * plan, and keeps the split-K partials in a static device array of
 * CONV_NOALLOC_SCRATCH_BYTES that is part of the library: every GPU that
 * loads the library holds that array until the process exits.  It calls no
 * cudaMalloc, cudaFree or allocating library routine.  The caller still
 * passes x, w, the scales and out.
 *   - A problem whose split-K partials need more than
 *     CONV_NOALLOC_SCRATCH_BYTES is rejected with CONV_ERR_INVALID
 *     (conv_last_error says how many bytes it needed), rather than run
 *     without split-K: a caller gets conv_fwd's plan or an error, never a
 *     silently slower plan.
 *   - Operand copies that conv_fwd makes in its workspace (aligned copies of
 *     a point-output GEMM's operands, the gathered rows of the patch class)
 *     go to the array too when they fit; the optional ones are skipped
 *     otherwise, while a patch-class problem whose gathered rows do not fit
 *     is rejected with CONV_ERR_INVALID.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept for the process, like
 *     the library's other per-device state (status word, copy streams): after
 *     cudaDeviceReset on a device, do not use the library on that device
 *     again in the same process.
 *   - Every call on a device shares the one array, which keeps the last
 *     call's contents.  Each call overwrites the partials it reads, so
 *     nothing needs clearing; but calls whose kernels overlap on the GPU
 *     (different streams, or threads racing on one device) race on the
 *     array and give wrong results.  Serialise them. */
int conv_fwd_noalloc(const void* x, const int64_t x_dims[5], const void* w,
                     const int64_t w_dims[5], const int stride[3], const int pad[3],
                     const int dil[3], int dtype, const float* scale_x, const float* scale_w,
                     void* out, cudaStream_t stream);

/* Plan and path overrides, for tile sweeps, A/B measurements and tests;
 * none is needed in normal use.  Every field set to -1 keeps the library's
 * own choice (conv_default_overrides fills a struct that way).  Nothing is
 * read from the environment: only conv_set_overrides changes these. */
typedef struct {
    int tile_n;          /* tile columns: 32..256, a multiple of 32 */
    int k_bytes;         /* bytes of one row per k-step: 32, 64, 128 or 256
                            (conv_fwd_ncdhw_fp8: 128 / 256 = one / two filter
                            taps per weight stage) */
    int stages;          /* shared-memory pipeline depth */
    int group_m;         /* raster group: consecutive m-tiles per group (>= 1) */
    int splits;          /* split-K factor (>= 1) */
    int pair;            /* 0: single CTAs, 1: CTA pairs (cta_group::2) */
    int msub;            /* row sub-tiles per unit sharing each B stage: 1 or 2 */
    int slices;          /* launches of whole waves a long reduction is cut into (>= 1) */
    int epilogue;        /* 1: TMA tensor stores, 2: staged 8/4-byte stores, 3: direct */
    int hw_major;        /* temporal class: 0 output-row order, 1 H*W-tile-major order */
    int two_phase;       /* point-output GEMM: 0 turns off the two-row-phase form */
    int repack;          /* point-output GEMM: 0 turns off the aligned operand copies */
    int dy_in_place;     /* backward weights: 0 transposes dy instead of reading it in place */
    int pdl;             /* 0: launches without programmatic dependent launch */
    int weight_groups;   /* conv_fwd_from_host: 0 keeps the first slice in one launch */
    int ncdhw_in_place;  /* conv_fwd_ncdhw: 1 always reads x in place (no packed copy) */
    int pack_lanes;      /* pack kernels: 2 or 4 lanes per position (warp-tile shape) */
    int log;             /* 1: print each plan and slice to stderr */
} conv_overrides;

/* Fills *o with -1 in every field (the library's own choices). */
void conv_default_overrides(conv_overrides* o);

/* Installs *o for every later call in the process; NULL restores the
 * defaults.  Returns CONV_ERR_INVALID (and keeps the previous overrides) for
 * a value outside a field's range.  Calls already enqueued are not
 * affected; calls running concurrently on other threads see either the old
 * or the new set. */
int conv_set_overrides(const conv_overrides* o);

/* Reads and clears the current device's status word, after synchronising
 * the device.  *device_status receives CONV_OK, or CONV_ERR_TIMEOUT if a
 * kernel gave up on a bounded wait since the last call.  Returns
 * CONV_ERR_CUDA if the synchronisation or copy failed. */
int conv_get_device_status(int* device_status);

/* conv_get_device_status in the order of one stream: after the work queued
 * on `stream` so far, reads and clears the current device's status word
 * and synchronises that stream only (not the device).  The word is shared
 * by every stream of the device, so a timeout recorded by a kernel on
 * another stream is reported (and cleared) here too.  Returns CONV_ERR_CUDA
 * if the copy or the synchronisation failed. */
int conv_get_device_status_stream(cudaStream_t stream, int* device_status);

/* Upper bound, in nanoseconds, on every spin-wait inside the kernels
 * (default 2e9 = 2 s).  A kernel that waits longer records CONV_ERR_TIMEOUT
 * in the device status word, drains its own copies in flight, frees its
 * tensor memory and returns.  Host-only setter; applies to later launches. */
void conv_set_wait_limit_ns(uint64_t ns);

/* Static description of a status code. */
const char* conv_status_string(int status);

/* Human-readable detail of the last non-OK return on the calling thread
 * (thread-local, overwritten by the next failure). */
const char* conv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* CONV3D_GB300_H */
