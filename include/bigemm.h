/*
 * bigemm.h -- C ABI of the broadcast / implicit-GEMM convolution library for
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * Operations (the sources that define them):
 *
 *  conv2d   NCHW 2-D convolution, as computed by topi.nn.conv2d_nchw in
 *           "Tuning High Performance Convolution on NVIDIA GPUs" (TVM v0.5
 *           autotvm tutorial), Step 1 (compute declaration, inlined padding):
 *             out[n,f,y,x] = sum_{rc<CI/groups, ry<KH, rx<KW}
 *                              pad(data)[n, g*CI/groups + rc, y*s+ry, x*s+rx]
 *                              * kernel[f, rc, ry, rx]
 *           with g = f / (CO/groups), pad() = `padding` zeros on every side,
 *           dilation 1, Ho = floor((H + 2*padding - KH)/stride) + 1 (Wo alike).
 *           The tutorial's template signature (N, H, W, CO, CI, KH, KW, stride,
 *           padding) gives the argument order of conv2d_nchw_plan.
 *  epilogue The per-channel broadcast of "[CINN] Add the TileBroadcastTactic
 *           for NCHW broadcast" (PaddlePaddle PR 70092), Introduction and
 *           Example, applied to the conv sum before the store:
 *             out[n,f,y,x] = op(acc[n,f,y,x] + bias[f]).
 *  bcast    The same PR's broadcast on its own:
 *             out[n,c,h,w] = op(var[c]),  [1,C,1,1] => [N,C,H,W],
 *           with the channel value computed once per channel block.
 *  plan     A timed choice among a few kernel tilings per shape, the analogue
 *           of the tutorial's Step 2 (tuning with a measure option of repeated
 *           timed runs, keeping the best record for the workload).
 *
 * Conventions for every entry point:
 *  * Tensors are contiguous and in the caller's DEVICE memory (pointers from
 *    cudaMalloc / torch): data [N,CI,H,W] (NCHW), kernel [CO,CI/groups,KH,KW]
 *    (OIHW), bias/var [C] fp32, out [N,CO,Ho,Wo] (NCHW).  The caller owns
 *    them; the library never frees or retains them past the call.
 *  * `stream` is a cudaStream_t (NULL = the legacy default stream).  Runs are
 *    asynchronous on it; only conv2d_nchw_plan with search=1 synchronises.
 *  * Every function returns a bigemm_status; none aborts or exits.  Shapes,
 *    dtypes and alignment are checked before any launch.  A launch failure
 *    returns BIGEMM_ERR_CUDA.  Kernels bound every wait; a wait that runs out
 *    sets a sticky device flag read by bigemm_last_device_error().
 *  * Plans own their scratch memory (packed operands, split-K partial sums),
 *    allocated by conv2d_nchw_plan and freed by conv2d_nchw_plan_destroy.
 *    Two runs of one plan must not overlap on the GPU (they share scratch).
 */
#ifndef BIGEMM_H
#define BIGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { BIGEMM_F32 = 0, BIGEMM_F16 = 1, BIGEMM_BF16 = 2 } bigemm_dtype;

/* Fused epilogue: out = acc (NONE), acc + bias[f] (BIAS),
 * exp(acc + bias[f]) (BIAS_EXP), 1/sqrt(acc + bias[f] + eps) (BIAS_RSQRT),
 * 1/(acc + bias[f]) (BIAS_RECIP, the div of the CINN broadcast page's complex
 * ops: div, exp, rsqrt), max(acc + bias[f], 0) (BIAS_RELU, add + ReLU). */
typedef enum {
    BIGEMM_EPI_NONE = 0,
    BIGEMM_EPI_BIAS = 1,
    BIGEMM_EPI_BIAS_EXP = 2,
    BIGEMM_EPI_BIAS_RSQRT = 3,
    BIGEMM_EPI_BIAS_RECIP = 4,
    BIGEMM_EPI_BIAS_RELU = 5
} bigemm_epilogue;

typedef enum {
    BIGEMM_OK = 0,
    BIGEMM_ERR_INVALID_ARG = 1,   /* bad shape, null pointer, misaligned buffer   */
    BIGEMM_ERR_UNSUPPORTED = 2,   /* valid conv this library does not implement  */
    BIGEMM_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed         */
    BIGEMM_ERR_TIMEOUT = 4,       /* a bounded device wait ran out               */
    BIGEMM_ERR_NO_CANDIDATE = 5   /* plan search found no runnable kernel        */
} bigemm_status;

/* Broadcast ops: out = var[c] (COPY), exp(var[c]) (EXP),
 * 1/sqrt(fp32(var[c] + eps)) (RSQRT), 1/var[c] (RECIP). */
typedef enum {
    BIGEMM_BC_COPY = 0,
    BIGEMM_BC_EXP = 1,
    BIGEMM_BC_RSQRT = 2,
    BIGEMM_BC_RECIP = 3
} bigemm_bcast_op;

/* Kernel families a plan can hold. */
typedef enum {
    BIGEMM_KIND_AUTO = 0,
    BIGEMM_KIND_UMMA = 1,         /* tcgen05 implicit GEMM (TF32 / FP16 / BF16)  */
    BIGEMM_KIND_SIMT = 2,         /* direct FP32-FMA conv (any shape, depthwise) */
} bigemm_kind;

typedef struct bigemm_plan_s *bigemm_plan;   /* opaque, library-owned */

/* Optional overrides for conv2d_nchw_plan_ex; zero fields mean "choose". */
typedef struct {
    int kind;       /* bigemm_kind                                              */
    int tile_n;     /* UMMA: output channels per tile, 16..256 step 16           */
    int split_k;    /* UMMA: number of K slices (>= 1)                          */
    int stages;     /* UMMA: shared-memory pipeline depth (2..8)                */
    int box_w;      /* UMMA: output pixels per tile along W (with box_h)        */
    int box_h;      /* UMMA: output rows per tile (box_w*box_h*boxes = 128);
                       SIMT depthwise: output rows per block of the staged-band
                       kernel (selects it over the streaming kernel)            */
    int mode;       /* UMMA operand-A mode: 1 channels-last boxes per tap,
                       2 NCHW read in place (1x1, stride 1, 16-bit),
                       3 one halo box per channel block (stride 1),
                       4 mode 1 over a subsampled copy (1x1, pad 0, stride > 1:
                         only the pixels the conv reads are packed),
                       5 mode 3 with the images stacked, pad zero rows apart,
                         so that one 16-row tile spans several small images,
                       6 NCHW read in place for a 1x1, stride-2, unpadded conv
                         (16-bit, H even, 2*W*element size a multiple of 16
                         bytes): TMA brings the even input rows, and warps of
                         the kernel keep the even pixels, so no packed copy is
                         made.
                       7 mode 1 with im2col tiles (K x K > 1, stride 1 or 2):
                         a tile is 128 consecutive output pixels of the
                         flattened N x Ho x Wo, across rows and images, and
                         each tap's operand is one TMA im2col load over the
                         channels-last copy (box_w and box_h are ignored;
                         outputs are written from registers).
                       With kind = SIMT it names the kernel instead: 1 tiled
                       (groups = 1) or naive, 2 depthwise staged band (box_h
                       rows per block), 3 depthwise streaming (box_h = 2, 4
                       or 8 rows per thread), 4 depthwise whole planes
                       (H, W <= 32, one or two planes per warp), 5 depthwise
                       small planes (stride 1, square 3/5/7 kernel, pad K/2,
                       outputs at most 16 wide and 32 tall; each thread
                       computes a box_h x 8 block of outputs, box_h = 2 or 4,
                       0 meaning 4), 6 depthwise bands of rows (square 3/5/7
                       kernel, pad K/2, stride 1 or 2, input rows whose bytes
                       are a multiple of 16 and at most 512; 4 x 8 outputs
                       per thread).
                       Other values: INVALID_ARG.                               */
    int resident_b; /* UMMA: 1 keeps the weights resident in shared memory --
                       halo modes: one output-channel tile must cover CO and
                       every tap must fit; other modes: split_k 1, and every K
                       block of one output-channel tile must fit (each block
                       keeps one tile) -- -1 streams them, 0 chooses            */
    int epi_warps;  /* UMMA modes 1, 2 and 4 with tile_n = 128: 16 runs four
                       epilogue warps per TMEM lane quadrant (576 threads per
                       block) instead of two (8); 0 chooses; other values:
                       INVALID_ARG                                              */
    int cta_pair;   /* UMMA modes 3 and 5 with resident weights, tile_n 64 or
                       128, split_k 1: 1 runs clusters of two blocks that share
                       each MMA (M = 256 pixels, each block holding half of the
                       weights), -1 single blocks, 0 chooses; other values:
                       INVALID_ARG                                              */
} bigemm_plan_options;

/*
 * conv2d_nchw_plan -- validate a conv shape and pick the kernel that runs it.
 *   N,H,W      batch and input spatial size (N >= 1, H, W >= 1)
 *   CO, CI     output / input channels; groups = 1, or groups = CI = CO
 *              (depthwise)
 *   KH, KW     kernel size; stride >= 1, padding >= 0 (dilation is 1)
 *   in_dtype   type of data and kernel: F32 (TF32 tensor cores or FP32 FMA),
 *              F16 or BF16 (fp32 accumulation)
 *   out_dtype  type of out (F32, F16 or BF16)
 *   epi        fused epilogue (bias is then required at run time)
 *   search     0: heuristic choice, no launch; 1: time every valid candidate
 *              with CUDA events on `stream` (synchronises) and keep the best
 *   out_plan   receives the plan; free it with conv2d_nchw_plan_destroy.
 * Errors: INVALID_ARG (Ho or Wo <= 0, bad groups, null out_plan),
 * UNSUPPORTED (e.g. depthwise with a channel multiplier), CUDA,
 * NO_CANDIDATE.  Plans are cached per (shape, dtypes, epilogue, device);
 * each call still returns a fresh handle.
 */
bigemm_status conv2d_nchw_plan(int N, int H, int W, int CO, int CI, int KH, int KW,
                               int stride, int padding, int groups,
                               bigemm_dtype in_dtype, bigemm_dtype out_dtype,
                               bigemm_epilogue epi, int search,
                               void *stream, bigemm_plan *out_plan);

/* As conv2d_nchw_plan, with optional overrides (opts may be NULL).  A forced
 * choice that cannot run this shape returns UNSUPPORTED.  Forced plans are
 * not cached. */
bigemm_status conv2d_nchw_plan_ex(int N, int H, int W, int CO, int CI, int KH, int KW,
                                  int stride, int padding, int groups,
                                  bigemm_dtype in_dtype, bigemm_dtype out_dtype,
                                  bigemm_epilogue epi, int search,
                                  const bigemm_plan_options *opts,
                                  void *stream, bigemm_plan *out_plan);

/*
 * conv2d_nchw_run -- run a plan on `stream`.
 *   data   [N,CI,H,W] device, in_dtype, 16-byte aligned
 *   kernel [CO,CI/groups,KH,KW] device, in_dtype, 16-byte aligned
 *   bias   [CO] fp32 device, or NULL when the plan's epilogue is NONE
 *   eps    added inside rsqrt for BIAS_RSQRT, ignored otherwise
 *   out    [N,CO,Ho,Wo] device, out_dtype, 16-byte aligned; fully written
 * Errors: INVALID_ARG (null or misaligned pointer, missing bias), CUDA.
 */
bigemm_status conv2d_nchw_run(bigemm_plan plan, const void *data, const void *kernel,
                              const float *bias, float eps, void *out, void *stream);

/* Free the plan and its scratch (synchronises with the device first). */
bigemm_status conv2d_nchw_plan_destroy(bigemm_plan plan);

/* Write a one-line JSON description of the plan (kernel, tiles, split-K,
 * launches per run, scratch bytes, search records) into buf (NUL-terminated,
 * truncated to len).  Returns INVALID_ARG for a NULL plan or buffer. */
bigemm_status conv2d_nchw_plan_describe(bigemm_plan plan, char *buf, size_t len);

/*
 * bcast_nchw_run -- out[n,c,h,w] = op(var[c]) for all n < N, h < H, w < W.
 *   var  [C] fp32 device; out [N,C,H,W] device of out_dtype (F32/F16/BF16).
 *   op   bigemm_bcast_op; eps is used by RSQRT only.
 * Errors: INVALID_ARG (N, C, H or W < 1, null pointer, bad op/dtype), CUDA.
 */
bigemm_status bcast_nchw_run(int N, int C, int H, int W, int op, const float *var, float eps,
                             void *out, bigemm_dtype out_dtype, void *stream);

/*
 * bcast_run -- the general form, out[b0,p,b1] = op(var[p]) for b0 < B0,
 * p < P, b1 < B1: any broadcast [1,P,1] => [B0,P,B1] after fusing adjacent axes
 * of the same kind, the last axis broadcast ("[CINN] Add the TileBroadcastTactic
 * for NCHW broadcast", PaddlePaddle PR 70092, Introduction).  The NCHW case is
 * B0 = N, P = C, B1 = H*W.  Long rows (B1 * element size >= 1 KB) run the
 * per-channel kernel of bcast_nchw_run; shorter rows a kernel whose threads
 * each own a fixed 16-byte piece of the P*B1 run and repeat it down B0.
 *   var  [P] fp32 device; out [B0,P,B1] device of out_dtype (F32/F16/BF16),
 *        aligned to its element size (16-byte alignment takes vector stores).
 *   op   bigemm_bcast_op; eps is used by RSQRT only.
 * Errors: INVALID_ARG (a size < 1, null pointer, bad op/dtype, misaligned
 * output), UNSUPPORTED (P*B1 > 2^31 - 1), CUDA.
 */
bigemm_status bcast_run(int B0, int P, int B1, int op, const float *var, float eps, void *out,
                        bigemm_dtype out_dtype, void *stream);

/* The same broadcast written the way a generic fused-loop schedule does it:
 * one flat loop over all N*C*H*W outputs, each recomputing op(var[c]) from
 * its own index.  Kept to measure the per-channel mapping against it. */
bigemm_status bcast_nchw_run_flat(int N, int C, int H, int W, int op, const float *var,
                                  float eps, void *out, bigemm_dtype out_dtype, void *stream);

/*
 * conv2d_nchw_run_noalloc -- the same convolution for callers that cannot
 * allocate device memory: code that runs where cudaMalloc is forbidden or
 * would break a memory budget someone else fixed, and so can neither create a
 * plan (plans own cudaMalloc'd scratch) nor lend the library a workspace.
 * The sources have no counterpart of this call; it exists for those callers.
 *
 * It runs the channels-last tensor-core kernel (the packed-operand path with
 * split-K when the tiles alone leave SMs idle) with every scratch byte in one
 * fixed array in the library's own device memory: 16 MiB (16777216 bytes),
 * held on every GPU that loads the library until the process exits.  The
 * scratch a shape needs is
 *   r(N*H*W*Ch*e) + r(CO*KH*KW*cip*e) + S*N*CO*Ho*Wo*4 bytes,
 * where r() rounds up to 256, e is the input element size, Ch = CI rounded up
 * to 16/e, cip = CI rounded up to 128/e, and S is the number of K slices.
 * S = 1 unless the pixel tiles times the channel tiles cover less than half
 * the SMs; then S is lowered, down to 1, until the partial sums fit.  Shapes
 * whose data and kernel copies alone exceed 16 MiB return
 * BIGEMM_ERR_UNSUPPORTED before any launch.
 *
 * Arguments and layouts are those of conv2d_nchw_plan + conv2d_nchw_run with
 * groups = 1 (data [N,CI,H,W], kernel [CO,CI,KH,KW], bias [CO] fp32, out
 * [N,CO,Ho,Wo], device pointers owned by the caller, 16-byte aligned;
 * stride <= 8).  timeout_flag is an optional device int the kernels set to 4
 * (BIGEMM_ERR_TIMEOUT) if a bounded device wait runs out (the caller clears
 * it); when NULL the kernels raise the library's sticky device flag instead,
 * which bigemm_last_device_error() reports and bigemm_clear_device_error()
 * clears.  That flag is a file-scope device variable too, not an allocation.
 *
 * The call allocates nothing: no cudaMalloc, cudaFree or allocating library
 * routine.  The first call on a device looks up the device address of the
 * scratch array (cudaGetSymbolAddress, with that device current), so make
 * that first call before any stream capture.  Every call on a device shares
 * the one array and leaves its contents behind; calls whose kernels overlap on
 * the GPU (different streams, or several host threads) race on it and must be
 * ordered by the caller.  Errors: INVALID_ARG (bad shape, dtype, epilogue,
 * null or misaligned pointer, missing bias), UNSUPPORTED (scratch above the
 * limit, stride > 8), CUDA.
 */
bigemm_status conv2d_nchw_run_noalloc(int N, int H, int W, int CO, int CI, int KH, int KW,
                                      int stride, int padding, bigemm_dtype in_dtype,
                                      bigemm_dtype out_dtype, bigemm_epilogue epi,
                                      const void *data, const void *kernel, const float *bias,
                                      float eps, void *out, int *timeout_flag, void *stream);

/* Human-readable text of a status code (static storage). */
const char *bigemm_status_string(bigemm_status s);

/* Sticky device-side flag: BIGEMM_ERR_TIMEOUT once any kernel's bounded wait
 * ran out on the current device (planned runs, broadcasts, and
 * conv2d_nchw_run_noalloc calls given no timeout_flag), else BIGEMM_OK.
 * Synchronises the device.  The flag is a file-scope device variable of the
 * library (one per device, zero at load), so reading it allocates nothing. */
bigemm_status bigemm_last_device_error(void);

/* Clear the sticky device flag (synchronises the device). */
bigemm_status bigemm_clear_device_error(void);

/* Upper bound, in nanoseconds, of every device-side wait of later launches
 * (default 2e9).  Values below 1000 are raised to 1000. */
bigemm_status bigemm_set_wait_timeout_ns(uint64_t ns);

/* Launch one block that waits on a barrier nothing will complete, bounded by
 * timeout_ns; the host then sees BIGEMM_ERR_TIMEOUT from
 * bigemm_last_device_error().  Exercises the timeout path without a fault. */
bigemm_status bigemm_debug_wait_timeout(uint64_t timeout_ns, void *stream);

/* Per-kernel timing with CUDA events recorded around each launch on its
 * stream.  enable(1) starts recording (and clears old records). */
typedef struct {
    char name[48];
    int launches;
    double total_ms;
} bigemm_kernel_time;

bigemm_status bigemm_profile_enable(int on);
/* Synchronises, then fills up to max entries; *count receives the number of
 * distinct kernels.  Records stay until the next enable(1). */
bigemm_status bigemm_profile_read(bigemm_kernel_time *out, int max, int *count);

/* Library version string. */
const char *bigemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BIGEMM_H */
