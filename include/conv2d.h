/*
 * conv2d.h — C ABI of the GB300 (sm_103a) forward 2-D convolution library.
 *
 * Operation (every entry point below computes or serves this):
 *
 *   Y[n,co,ho,wo] = sum_{ci,kh,kw} X[n,ci, ho*s+kh-p, wo*s+kw-p] * W[co,ci,kh,kw]
 *
 * a cross-correlation (no kernel flip) with symmetric zero padding p and one
 * stride s, as defined in "Enabling Memory-efficient Im2win Convolution with
 * Multi-precision Support on GPU CUDA and Tensor Cores", Sec. III-A, Eq. (1),
 * and in the 7-loop of "Unifying Convolutions and GEMM", Sec. 1.  Output size
 * (floor rule, "Unifying Convolutions and GEMM", Sec. 5):
 *
 *   Ho = (H + 2p - Kh) / s + 1,   Wo = (W + 2p - Kw) / s + 1.
 *
 * Conventions for every call:
 *   - All functions return a conv2d_status; no C++ exception crosses the ABI.
 *   - Device pointers are plain CUDA device addresses owned by the caller.
 *     The library never allocates, frees or retains device memory, and keeps
 *     no pointer after a call returns, except the bias pointer a caller sets
 *     on a descriptor (conv2d_desc_set_bias), which that descriptor's calls
 *     read.
 *   - `stream` is a cudaStream_t (or CUstream) cast to void*; NULL is the
 *     legacy default stream.  Kernels are launched asynchronously on it;
 *     conv2d_fwd returns once the launches are queued.
 *   - A descriptor is immutable after creation except through the
 *     conv2d_desc_set_* calls; concurrent conv2d_fwd calls on one descriptor
 *     from several host threads are safe (each call uses only its arguments).
 */
#ifndef CONV2D_GB300_H
#define CONV2D_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONV2D_OK = 0,
    CONV2D_ERR_BAD_PARAM = 1,            /* invalid geometry or enum value              */
    CONV2D_ERR_UNSUPPORTED = 2,          /* valid request this build does not implement */
    CONV2D_ERR_NULL_PTR = 3,             /* a required pointer was NULL                 */
    CONV2D_ERR_MISALIGNED = 4,           /* a device pointer was not 16-byte aligned    */
    CONV2D_ERR_WORKSPACE_TOO_SMALL = 5,  /* workspace_bytes < conv2d_workspace_size     */
    CONV2D_ERR_CUDA = 6,                 /* a CUDA runtime/driver call failed           */
    CONV2D_ERR_DEVICE_TIMEOUT = 7        /* a kernel's bounded wait expired (see below) */
} conv2d_status;

/* Element type of X and W.  Accumulation is always fp32 (fp32 FFMA on the
 * CUDA-core path, fp32 TMEM accumulators on the tensor-core path).  Y is fp32
 * for CONV2D_F32 and has the input type for CONV2D_F16 / CONV2D_BF16, rounded
 * to nearest even once at the store. */
typedef enum { CONV2D_F32 = 0, CONV2D_F16 = 1, CONV2D_BF16 = 2 } conv2d_dtype;

/* Algorithms.
 *  IM2WIN_FP32_CC   fp32 on CUDA cores.  Workspace holds the im2win tensor of
 *                   "Enabling Memory-efficient Im2win Convolution ...",
 *                   Sec. III-B, Eq. (2) (one strip of Kh rows per output row
 *                   and input channel, padding included); the convolution of
 *                   Sec. III-C, Eq. (3) reads it.
 *  IM2WIN_TC        fp16/bf16 on tcgen05 tensor cores.  Workspace holds the
 *                   channels-innermost window tensor (the NHWC variant the
 *                   same paper uses on tensor cores, Sec. III-D) and the
 *                   repacked filter.
 *  IMPLICIT_TC      fp16/bf16 on tcgen05 tensor cores; operand tiles are
 *                   gathered straight from channels-last X in the load path
 *                   (the implicit expansion of "im2col Expansion, FFT
 *                   Convolution, and Winograd Transforms", im2col section).
 *                   Workspace: the repacked filter, plus a channels-last copy
 *                   of X when the input layout is NCHW.  A 1x1, stride-1,
 *                   unpadded layer on NCHW input with Cin and H*W multiples
 *                   of 8 is one GEMM per image, Y[co][p] = sum_ci W[co][ci]
 *                   X[ci][p] (the convolution sum with Kh = Kw = 1, s = 1,
 *                   p = 0, where the expansion is the identity): it reads x
 *                   and w in place, needs no workspace (size 0) and makes
 *                   one launch.
 *  IMPLICIT_FP32_CC fp32 on CUDA cores, staging X's rows directly (no input
 *                   expansion); workspace: the repacked filter only.
 *  PADDED_TC        fp16/bf16 on tcgen05 tensor cores, stride 1 and NCHW input
 *                   only.  X is copied once into a zero-padded channels-last
 *                   buffer; the GEMM rows walk the padded grid, so each filter
 *                   tap's operand tile is one tiled TMA box at a constant
 *                   shift (kh*pitch + kw) and the outputs at padded positions
 *                   are discarded.  Workspace: repacked filter + padded copy.
 *  IMPLICIT_NCHW_TC fp16/bf16 on tcgen05 tensor cores, stride 1, NCHW input:
 *                   the implicit expansion done inside the contraction kernel
 *                   with no copy of X ("im2col Expansion, FFT Convolution, and
 *                   Winograd Transforms", im2col section: the indexing lives
 *                   in the GEMM's load path).  The kernel reads X in place and
 *                   builds each zero-padded channels-last operand tile in
 *                   shared memory; every tap of a filter-row group reads that
 *                   tile at a row offset.  Workspace: the repacked filter
 *                   only; two launches (repack, contraction).
 *  WINOGRAD_FP32_CC fp32 on CUDA cores, 3x3 filters at stride 1 (any pad),
 *                   NCHW input: Winograd minimal filtering F(2x2, 3x3)
 *                   ("OpenCNN: a Winograd minimal filtering algorithm
 *                   implementation in CUDA", Sec. 2-3; "im2col Expansion,
 *                   FFT Convolution, and Winograd Transforms", Winograd
 *                   section): a filter-transform kernel, then one kernel per
 *                   call that transforms 4x4 input tiles, sums the 16
 *                   transformed products over input channels and transforms
 *                   each 2x2 output tile back.  2.25x fewer multiplications
 *                   than the direct sum; the same fp32 parity contract.
 *                   Workspace: the transformed filter (16 values per filter,
 *                   input channels rounded up to 8, output channels to 64).
 *  AUTO             resolved per shape when the descriptor is created
 *                   (conv2d_get_algo reports the choice). */
typedef enum {
    CONV2D_ALGO_AUTO = 0,
    CONV2D_ALGO_IM2WIN_FP32_CC = 1,
    CONV2D_ALGO_IM2WIN_TC = 2,
    CONV2D_ALGO_IMPLICIT_TC = 3,
    CONV2D_ALGO_IMPLICIT_FP32_CC = 4,
    CONV2D_ALGO_PADDED_TC = 5,
    CONV2D_ALGO_IMPLICIT_NCHW_TC = 6,
    CONV2D_ALGO_WINOGRAD_FP32_CC = 7
} conv2d_algo;

/* Memory layout of X.  Y is always NCHW.  W is always [Cout][Cin][Kh][Kw]. */
typedef enum { CONV2D_LAYOUT_NCHW = 0, CONV2D_LAYOUT_NHWC = 1 } conv2d_layout;

typedef struct conv2d_desc *conv2d_desc_t;   /* opaque, host memory, owned by the caller */

/* Create a descriptor for one problem shape.  Host-only: makes no CUDA call,
 * so it works without a GPU.  Arguments follow the problem statement of
 * "Enabling Memory-efficient Im2win Convolution ...", Sec. III-A (N, Ci, Hi,
 * Wi, Co, Hf, Wf, s) with the padding of "Unifying Convolutions and GEMM",
 * Sec. 5.
 *   out       receives the new descriptor (set to NULL on failure)
 *   N, Cin, H, W   input batch, channels, height, width   (all >= 1)
 *   Cout           output channels                         (>= 1)
 *   Kh, Kw         filter height and width                 (>= 1)
 *   stride >= 1, pad >= 0 (symmetric, zero fill); Ho and Wo must be >= 1
 *   dtype, algo    see above; an algo that does not serve dtype -> BAD_PARAM
 * Errors: NULL_PTR (out NULL), BAD_PARAM (any check above, or a tensor with
 * more than 2^31-1 elements), UNSUPPORTED (shape outside the algo's limits,
 * e.g. pad > 127 on a tensor-core algo). */
conv2d_status conv2d_desc_create(conv2d_desc_t *out, int N, int Cin, int H, int W, int Cout,
                                 int Kh, int Kw, int stride, int pad,
                                 conv2d_dtype dtype, conv2d_algo algo);

/* Select the layout of X (default NCHW).  Re-resolves AUTO and changes the
 * workspace size; call before conv2d_workspace_size.  BAD_PARAM for an
 * unknown layout; UNSUPPORTED for NHWC with an fp32 algorithm. */
conv2d_status conv2d_desc_set_input_layout(conv2d_desc_t d, conv2d_layout layout);

/* Element type of Y.  Default: the input dtype (fp16/bf16 outputs rounded to
 * nearest even once, from the fp32 accumulator).  For CONV2D_F16 /
 * CONV2D_BF16 inputs, CONV2D_F32 keeps the fp32 accumulator unrounded (Y is
 * then [N][Cout][Ho][Wo] floats).  The pages fix no output type for 16-bit
 * inputs ("Enabling Memory-efficient Im2win Convolution ...", Sec. III-F
 * says only that the tensor cores take fp16); this option serves callers
 * that want the fp32 sum.  BAD_PARAM for any other type. */
conv2d_status conv2d_desc_set_output_dtype(conv2d_desc_t d, conv2d_dtype out);

/* Per-output-channel bias, the `Y_col += bias` of the PyTorch listing in
 * "Unifying Convolutions and GEMM", Sec. 6:
 *   Y[n,co,ho,wo] = b[co] + sum_{ci,kh,kw} X[...] * W[...]
 * added to the fp32 accumulator before the one rounding to Y's type.
 *   bias  device pointer to Cout elements of the INPUT dtype (fp32 for
 *         CONV2D_F32, else fp16/bf16 like W), or NULL for no bias (default).
 * The descriptor keeps the pointer (it does not copy the values): every
 * conv2d_fwd* call made with this descriptor reads b from it on the GPU, so
 * the buffer must stay valid while such calls can run.  Errors: NULL_PTR (d),
 * MISALIGNED (bias not aligned to its element size). */
conv2d_status conv2d_desc_set_bias(conv2d_desc_t d, const void *bias);

/* Knobs of the pipeline, for ablation studies in the manner of "Enabling
 * Memory-efficient Im2win Convolution ...", Sec. IV-E (Fig. 4: the kernel
 * without double buffering, without asynchronous copies, without the
 * zig-zag block order).  Results do not depend on them (same sums; only the
 * order in which tiles are visited and copies overlap changes).
 *   CONV2D_TUNE_STAGES        cap on the depth of the shared-memory operand
 *                             ring: 1 = no double buffering (every stage's
 *                             copies wait for the previous stage's MMAs or
 *                             FMAs), 2..8, 0 = automatic (default).  The
 *                             CUDA-core kernel has two stages: 1 selects one.
 *   The other knobs act on the tensor-core kernels only.
 *   CONV2D_TUNE_SYNC_COPIES   1 = the copy-issuing thread waits for each
 *                             stage's copies to land before it issues the
 *                             next stage (copies no longer overlap each
 *                             other); 0 = asynchronous (default).
 *   CONV2D_TUNE_RASTER        visit order of the output tile groups (tensor
 *                             cores): 0 = output-channel tile fastest
 *                             (default), 1 = pixel group fastest, 2 = zig-zag
 *                             (channel tiles in alternating direction on
 *                             successive pixel groups).
 *   CONV2D_TUNE_NO_RESIDENT   1 = never keep the filter slice resident in
 *                             shared memory (tensor cores); 0 = automatic.
 *   CONV2D_TUNE_SPLIT         1 = when the output tiles do not divide evenly
 *                             over the SMs, split the filter-tap stages of the
 *                             last, partial wave evenly over all SMs; each
 *                             tile's first SM adds the others' fp32 partial
 *                             sums (published through the workspace) before
 *                             its epilogue, so only the order of the sum
 *                             changes.  Needs more workspace (fp32 partials
 *                             for up to one tile per SM; conv2d_workspace_size
 *                             includes it when the split will run and the
 *                             total stays within the im2win tensor).  0 = the
 *                             last wave takes whole tiles (default: on GB300
 *                             a last wave of whole tiles runs faster per SM
 *                             than a full one, and the owners' additions
 *                             give back most of the balance, so the split
 *                             measured at best 1 % faster and often slower).
 *                             UNSUPPORTED while a 176-wide tile is
 *                             requested (CONV2D_TUNE_TILE_N); the automatic
 *                             width then keeps to 64, 128 or 256.
 *   CONV2D_TUNE_EPI_GROUPS    warps that store the output (tensor cores,
 *                             implicit, padded and im2win sources): 2 = two
 *                             groups of four warps, 3 = three groups with a
 *                             third accumulator buffer per MMA issuer (output
 *                             tiles up to 128 channels wide; 128-wide tiles
 *                             then run one per MMA issuer), 0 = automatic
 *                             (default).  Ignored when the split runs.
 *   CONV2D_TUNE_TILE_N        output channels per tensor-core tile: 64, 128,
 *                             176 or 256 (176 on the implicit, padded and
 *                             im2win sources only, not with the split), 0 =
 *                             automatic (default: the width that needs the
 *                             fewest waves of tile groups).  1x1 layers keep
 *                             128.  Errors: UNSUPPORTED when the width does
 *                             not apply to the descriptor's algorithm.
 * Errors: NULL_PTR, BAD_PARAM (unknown knob or value out of range). */
typedef enum {
    CONV2D_TUNE_STAGES = 0,
    CONV2D_TUNE_SYNC_COPIES = 1,
    CONV2D_TUNE_RASTER = 2,
    CONV2D_TUNE_NO_RESIDENT = 3,
    CONV2D_TUNE_SPLIT = 4,
    CONV2D_TUNE_EPI_GROUPS = 5,
    CONV2D_TUNE_TILE_N = 6
} conv2d_tuning;
conv2d_status conv2d_desc_set_tuning(conv2d_desc_t d, conv2d_tuning knob, int value);

/* Pre-packed filters.  Every call repacks the filter into the order its
 * kernels read (the filter-height-before-width, channel-innermost order of
 * "Enabling Memory-efficient Im2win Convolution ...", Sec. III-C/III-D; the
 * transformed filter G g G^T for Winograd).  A caller whose filter does not
 * change between calls (inference) can pack it once:
 *   conv2d_packed_filter_bytes  size of the packed filter for the
 *                               descriptor's algorithm (bytes)
 *   conv2d_pack_filter          w (the [Cout][Cin][Kh][Kw] filter, device)
 *                               -> w_packed (device, that many bytes, 16-byte
 *                               aligned), on `stream`
 *   conv2d_desc_set_filter_prepacked(d, 1)
 *                               from then on conv2d_fwd* take w_packed as
 *                               their w argument: no repack launch, and
 *                               conv2d_workspace_size no longer includes the
 *                               packed filter.  0 restores the default.
 * The packed layout depends on the descriptor's shape and algorithm only;
 * pack again after changing either (a new descriptor).  Errors: NULL_PTR,
 * MISALIGNED, CUDA; BAD_PARAM for a flag other than 0/1. */
conv2d_status conv2d_packed_filter_bytes(conv2d_desc_t d, size_t *bytes);
conv2d_status conv2d_pack_filter(conv2d_desc_t d, const void *w, void *w_packed, void *stream);
conv2d_status conv2d_desc_set_filter_prepacked(conv2d_desc_t d, int prepacked);

/* Release a descriptor (NULL is accepted and ignored). */
conv2d_status conv2d_desc_destroy(conv2d_desc_t d);

/* Output spatial size (floor rule above). */
conv2d_status conv2d_out_dims(conv2d_desc_t d, int *Ho, int *Wo);

/* Workspace bytes conv2d_fwd needs for the resolved algorithm (may be 0).
 * The buffer must be device memory, 16-byte aligned (256 recommended). */
conv2d_status conv2d_workspace_size(conv2d_desc_t d, size_t *bytes);

/* Algorithm the descriptor resolved to (never AUTO). */
conv2d_status conv2d_get_algo(conv2d_desc_t d, conv2d_algo *chosen);

/* Forward convolution on `stream`.
 *   x  device, layout per conv2d_desc_set_input_layout, dtype of the desc
 *   w  device, [Cout][Cin][Kh][Kw] contiguous, dtype of the desc
 *   y  device, [N][Cout][Ho][Wo] contiguous, of the output dtype (the input
 *      dtype unless conv2d_desc_set_output_dtype chose fp32); plus b[co]
 *      when conv2d_desc_set_bias gave a bias
 *   workspace, workspace_bytes: device scratch of at least
 *      conv2d_workspace_size bytes (NULL/0 allowed when that size is 0);
 *      its contents on entry do not matter and are garbage on exit.
 * x, w, y and workspace must be 16-byte aligned and must not overlap y.
 * Errors: NULL_PTR, MISALIGNED, WORKSPACE_TOO_SMALL (checked before any
 * launch), CUDA (a launch or driver call failed; the CUDA error is left
 * pending for the caller to inspect).  Device-side timeouts are reported by
 * conv2d_device_status, not here, because launches are asynchronous. */
conv2d_status conv2d_fwd(conv2d_desc_t d, const void *x, const void *w, void *y,
                         void *workspace, size_t workspace_bytes, void *stream);

/* conv2d_fwd that also records two CUDA events on `stream`: `ev_start`
 * immediately before and `ev_end` immediately after the launch of the main
 * contraction kernel (the im2win / implicit-GEMM / CUDA-core convolution
 * kernel, not the transforms).  Events are cudaEvent_t cast to void*; either
 * may be NULL.  Lets a caller time that kernel alone inside a full call.
 * Same arguments, layouts and errors as conv2d_fwd, plus CONV2D_ERR_CUDA when
 * an event record fails. */
conv2d_status conv2d_fwd_profiled(conv2d_desc_t d, const void *x, const void *w, void *y,
                                  void *workspace, size_t workspace_bytes, void *stream,
                                  void *ev_start, void *ev_end);

/* conv2d_fwd for operands in host memory.  On `stream`, in order: copies
 * x_host into x_dev and w_host into w_dev (one cudaMemcpyAsync each), runs
 * conv2d_fwd(d, x_dev, w_dev, y_dev, workspace, ...), and copies y_dev back
 * into y_host.  Sizes follow the descriptor: x holds N*Cin*H*W and w
 * Cout*Cin*Kh*Kw elements of the input dtype (in the descriptor's input
 * layout), y N*Cout*Ho*Wo elements of the output dtype.  The caller owns all
 * buffers; the device ones obey conv2d_fwd's rules.  With page-locked host
 * memory the call returns before the copies finish (synchronise the stream
 * before reading y_host or reusing x_host); with pageable memory the CUDA
 * runtime stages the copies.  Calls on different streams overlap, so a caller
 * streaming batches can hide one call's copies behind another's compute.
 * Errors: as conv2d_fwd (checked before any copy), NULL_PTR for a null host
 * pointer, CUDA when a copy cannot be issued. */
conv2d_status conv2d_fwd_host(conv2d_desc_t d, const void *x_host, const void *w_host, void *y_host,
                              void *x_dev, void *w_dev, void *y_dev, void *workspace,
                              size_t workspace_bytes, void *stream);

/* Number of kernel launches one conv2d_fwd call makes for this descriptor
 * (filter repack, input transform if any, contraction; the contraction alone
 * for the in-place 1x1 GEMM). */
conv2d_status conv2d_launches_per_call(conv2d_desc_t d, int *launches);

/* Size of the library's built-in workspace used by
 * conv2d_fwd_static_workspace (64 MiB). */
#define CONV2D_STATIC_WORKSPACE_BYTES (64u << 20)

/* conv2d_fwd for callers that cannot allocate device memory (a host
 * application that owns all device memory and passes in only the tensors, a
 * loop that cannot afford the synchronisation of cudaMalloc/cudaFree, a
 * process under a memory cap set by someone else).  The paper has no
 * counterpart to this call; it is a deployment convenience.
 *   Same x, w, y, stream and layouts as conv2d_fwd; no workspace argument:
 *   scratch comes from one array of CONV2D_STATIC_WORKSPACE_BYTES that is
 *   part of the library's device image on every GPU that loads the library,
 *   held until the process exits.  The call allocates nothing.
 *   The first call on each device (with that device current) looks up the
 *   array's device address; make that first call before any stream capture.
 *   The address is then kept for the life of the process, which assumes the
 *   device's primary context is never destroyed (no cudaDeviceReset between
 *   calls): a reset context may load the array at another address.
 *   Every call uses the same array and it keeps the previous call's contents
 *   (nothing in it needs to start at zero).  Calls whose kernels overlap on
 *   the GPU (other streams, other host threads) race on it: serialise them.
 * Errors: as conv2d_fwd; WORKSPACE_TOO_SMALL when conv2d_workspace_size(d)
 * exceeds CONV2D_STATIC_WORKSPACE_BYTES (checked before any launch); CUDA
 * when the address lookup fails. */
conv2d_status conv2d_fwd_static_workspace(conv2d_desc_t d, const void *x, const void *w, void *y,
                                          void *stream);

/* Size in bytes of the array conv2d_fwd_static_workspace uses
 * (CONV2D_STATIC_WORKSPACE_BYTES of the library as built), for bindings that
 * cannot read the macro.  Errors: NULL_PTR. */
conv2d_status conv2d_static_workspace_bytes(size_t *bytes);

/* Read and clear the library's device status word on the current device
 * (synchronises `stream`).  Returns CONV2D_OK when every kernel since the
 * last call finished normally, CONV2D_ERR_DEVICE_TIMEOUT when a kernel gave
 * up on a bounded wait (its output is then invalid), CONV2D_ERR_CUDA when the
 * readback failed.  `*code_out` (may be NULL) receives the raw status bits. */
conv2d_status conv2d_device_status(void *stream, uint32_t *code_out);

/* Limit, in nanoseconds, of each pipeline wait of the library's kernels on
 * the current device (default 2 s, which is also the maximum: ns = 0 or a
 * value above it gives the default), for
 * kernels launched on `stream` after this call returns (the call
 * synchronises `stream`).  A wait that runs past the limit gives up: the
 * kernel lets the copies and MMAs it already issued finish, exits, and sets
 * the bit conv2d_device_status reports as CONV2D_ERR_DEVICE_TIMEOUT (that
 * call's output is invalid).  A tiny limit makes ordinary waits give up, so
 * a test can check this path without any wait that never ends.  Not for
 * production use.  The paper has no counterpart.  Errors: CUDA. */
conv2d_status conv2d_set_wait_limit(uint64_t ns, void *stream);

/* Static string for a status code (never NULL). */
const char *conv2d_status_string(conv2d_status s);

#ifdef __cplusplus
}
#endif
#endif /* CONV2D_GB300_H */
