/*
 * dl_linear.h -- C ABI of the GB300 (sm_103a) decode-linear library.
 *
 * The operation (one decode linear layer):
 *
 *     y[m][n] = bias[n] + sum_k x[m][k] * w(n, k),   0 <= m < M <= 16
 *
 * with bf16 activations x[M][K], weights stored [N][K] (K contiguous), fp32
 * accumulation and bf16 output rounded once, to nearest even.  This is the
 * tall-skinny decode GEMV/GEMM of "Developing a custom Qwen2.5 72B inference
 * engine from scratch" (§6.1 "Decode GEMV: already near the roofline": a
 * memory-bound matrix times a token vector, measured by the fraction of peak
 * HBM bandwidth it reaches; §2: every decoded token streams every weight once)
 * and of "9% faster GLM-5.3-Flash prefill with GPU-to-GPU IPC" (section
 * "TileLang: twice as fast, and no faster": a ~6-token verify step, 16-bit
 * activations, weight-only FP8 with one scale per 128x128 block, the long K
 * dimension split across blocks so that the whole chip streams weights).
 *
 * w(n, k) is either the bf16 weight W[n][k], or, for weight-only FP8,
 * e4m3(Wq[n][k]) * scales[n / 128][k / 128]: each e4m3 weight (OCP E4M3FN,
 * decoded exactly) times the fp32 scale of the 128x128 block it lies in, the
 * dequantisation of the same TileLang section, where the weight tile is
 * multiplied by its block's scale before the 16-bit GEMM.  Activations are
 * never quantised (weight-only FP8; same engine page, §6.2).
 *
 * Conventions for every entry point below:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    owned by the caller.  The library keeps no reference after a call
 *    returns and allocates no device memory on any call path.
 *  - Every tensor is dense and row-major exactly as described; there are no
 *    stride arguments.
 *  - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t
 *    passed as void*; NULL = the legacy default stream) and the host is never
 *    synchronised.  Results are valid once the stream has reached the call.
 *  - All arguments are validated BEFORE anything is enqueued.  On a non-OK
 *    status nothing was launched and nothing was written; dl_last_error()
 *    returns a message for the calling thread.  No C++ exception crosses the
 *    ABI.
 *  - Shapes: 1 <= M <= 16; 1 <= N, K < 2^31; BF16 needs K % 8 == 0 and FP8
 *    needs K % 128 == 0 (else DL_ERR_UNSUPPORTED_SHAPE).  x and W/Wq must be
 *    16-byte aligned (DL_ERR_MISALIGNED); bias/y 2-byte, y_f32/scales 4-byte.
 *  - Shapes also need N <= 2,097,152 (16,384 tiles of 128 rows).
 *  - Workspace: a device buffer of at least dl_workspace_bytes(...) bytes
 *    (256-byte aligned) whose first DL_WORKSPACE_ZERO_BYTES are ZERO-FILLED
 *    ONCE before its first use: the arrival counters, which every call returns
 *    to zero, so they never need clearing again unless a call reported a
 *    device-side error.  The rest is scratch (split-K partial sums and, for
 *    FP8, an f16 copy of x) that every call writes before it reads.  One
 *    workspace serves calls of any shape in turn; two calls that may run at
 *    the same time (different streams) must not share a workspace.
 *  - Results are deterministic: the same inputs, shape, device (SM count) and
 *    overrides give bitwise identical outputs on every call.
 */
#ifndef DL_LINEAR_H
#define DL_LINEAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DL_VERSION 3

/* Leading workspace bytes that must be zero before a call (see conventions). */
#define DL_WORKSPACE_ZERO_BYTES (256u + 16384u * 4u)

typedef enum dl_status {
    DL_OK = 0,
    DL_ERR_INVALID_ARG = 1,        /* NULL pointer, bad enum, negative size      */
    DL_ERR_UNSUPPORTED_SHAPE = 2,  /* M outside [1,16], K not a multiple of 8/128 */
    DL_ERR_MISALIGNED = 3,         /* a pointer breaks its alignment rule         */
    DL_ERR_WORKSPACE = 4,          /* workspace NULL or smaller than required     */
    DL_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed           */
    DL_ERR_DEVICE = 6              /* a kernel reported an error (dl_device_status) */
} dl_status;

/* Weight formats. */
typedef enum dl_dtype {
    DL_BF16 = 0,       /* W: bf16 [N][K]                                       */
    DL_FP8_B128 = 1    /* Wq: e4m3 codes [N][K] + fp32 scales [ceil(N/128)][K/128] */
} dl_dtype;

/* Kernel families (for dl_set_override; DL_KERNEL_AUTO picks by dtype and M). */
typedef enum dl_kernel {
    DL_KERNEL_AUTO = 0,
    DL_KERNEL_SIMT = 1,   /* CUDA-core FMA, one weight row per lane (FP8: M <= 2;
                             larger M runs the MMA family)                    */
    DL_KERNEL_MMA = 2,    /* warp-level tensor-core MMA (mma.sync): bf16, or f16
                             for FP8 weights against an exact f16 copy of x    */
    DL_KERNEL_TC = 3      /* FP8 weights only (bf16 layers keep their automatic
                             family): 5th-generation tensor cores, tcgen05.mma
                             kind::f8f6f4 with the e4m3 weight tile read from
                             shared memory as is, x split exactly into three
                             e4m3 parts, fp32 accumulators in tensor memory   */
} dl_kernel;

/*
 * Bytes of workspace one call with this shape needs on the current device
 * (it depends on the SM count and on any override set).  Returns 0 for an
 * invalid shape or dtype.  Never launches anything.
 */
size_t dl_workspace_bytes(int M, int N, int K, int dtype);

/*
 * y = x . W^T (+ bias), bf16 weights.
 *   x      bf16 [M][K], 16-byte aligned (K % 8 == 0 keeps every row aligned)
 *   W      bf16 [N][K], 16-byte aligned
 *   bias   bf16 [N] or NULL; added once in fp32 after the full K sum
 *   y      bf16 [M][N]; written (round to nearest even, once)
 *   y_f32  fp32 [M][N] or NULL; receives the value before rounding, so that
 *          y == RNE_bf16(y_f32) bit for bit (a test/debug output)
 *   workspace, ws_bytes: see the conventions above
 *   stream cudaStream_t
 */
dl_status dl_linear_bf16(const void* x, const void* W, const void* bias, void* y,
                         float* y_f32, int M, int N, int K, void* workspace,
                         size_t ws_bytes, void* stream);

/*
 * y = x . dequant(Wq)^T (+ bias), weight-only FP8 with 128x128 block scales.
 *   Wq     e4m3 (E4M3FN) codes [N][K] as bytes, 16-byte aligned, K % 128 == 0
 *   scales fp32 [ceil(N/128)][K/128] row-major: scales[n/128][k/128], 4-byte
 *          aligned; the kernel copies them in 16-byte-aligned pieces, so it
 *          may also read up to 12 bytes just before scales[0] (the rest of
 *          that 16-byte block, always in the same page), never after the end
 *   other arguments as for dl_linear_bf16.
 * Each e4m3 code is decoded exactly (NaN codes 0x7F/0xFF decode to NaN); the
 * block scale multiplies the fp32 partial sum of each 128-wide K block, which
 * is algebraically the same as scaling every weight.
 * Enqueues two kernels: an activation prep kernel (writes the exact f16 copy
 * of x into the workspace) and the main kernel.  If the second launch fails
 * (DL_ERR_CUDA), the first may have run; it writes only the workspace.
 */
dl_status dl_linear_fp8_block128(const void* x, const void* Wq, const float* scales,
                                 const void* bias, void* y, float* y_f32, int M, int N,
                                 int K, void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of the library's static device scratch (see below): 16 MiB per device.
 */
#define DL_STATIC_SCRATCH_BYTES (16u << 20)

/*
 * dl_linear_bf16 without a caller-supplied workspace: the split-K scratch is a
 * file-scope device array of DL_STATIC_SCRATCH_BYTES inside the library, and
 * neither this function nor anything it calls allocates device memory (no
 * cudaMalloc, no cudaFree, no allocating library routine).
 *
 * Who needs it: code that may not allocate device memory of its own -- for
 * instance a plugin running inside a host framework whose allocator owns the
 * whole device-memory budget, or a latency-critical decode loop that must not
 * call cudaMalloc/cudaFree because they can synchronise the device and stall
 * every other stream.
 *
 * The pages that define the operation have no counterpart to this entry point;
 * it is an interface convenience, computing exactly what dl_linear_bf16 does.
 *
 * Arguments: as for dl_linear_bf16, minus workspace/ws_bytes.
 * Limits and errors: shapes whose work plan needs more than
 *   DL_STATIC_SCRATCH_BYTES of scratch (dl_workspace_bytes(M, N, K, DL_BF16)
 *   tells) are rejected with DL_ERR_WORKSPACE before anything is enqueued.  The
 *   limit covers every Qwen2.5-72B decoder linear and the lm_head at M <= 8.
 * Set-up and cost: the array is part of the library's device code, so every
 *   process that loads the library reserves DL_STATIC_SCRATCH_BYTES on each
 *   device where that code is loaded -- whether or not it ever calls this
 *   entry point -- until the process exits.  With CUDA's lazy module loading
 *   (the default) the code, and so the array, may be placed on a device only
 *   by the first call that needs it, possibly this entry point's first call.
 *   That first call on each device, with that device current, also looks up
 *   the array's device address (cudaGetSymbolAddress) and caches it per device
 *   index.  Make that first call outside latency-critical code and before any
 *   stream capture begins.  The cached address does not survive a context
 *   reset (cudaDeviceReset): do not call this entry point on a device after
 *   resetting it in the same process.
 * Sharing: every call on a device uses the same array, which keeps what the
 *   last call left.  Each call first clears (cudaMemsetAsync on `stream`) the
 *   arrival counters that must start at zero; the partial sums need no
 *   clearing.  Calls ordered on one stream are safe; calls that can overlap on
 *   the GPU (other streams, other threads) race on the array and give wrong
 *   results.  If the kernel launch itself fails (DL_ERR_CUDA), that clearing
 *   may already be enqueued; it touches only the library's array.
 */
dl_status dl_linear_bf16_static_scratch(const void* x, const void* W, const void* bias, void* y,
                                        float* y_f32, int M, int N, int K, void* stream);

/*
 * gate_up projection with the SwiGLU activation fused into its epilogue:
 *     y[m][j] = silu(g) * u,   silu(g) = g / (1 + e^-g),
 * g and u the full fp32 sums (+ bias) of the gate and up rows of output j,
 * evaluated in fp32 and rounded once to bf16.  This is the nonlinearity
 * between the two matrices of the MLP in "Multi-GPU Inference and Serving at
 * Scale", Example 3 (shown there as a ReLU; the page names SwiGLU as the
 * variant real models use), in its usual SiLU-gated form.
 *   dtype  DL_BF16 or DL_FP8_B128 (as for the plain calls; FP8 scales cover
 *          128x128 blocks of W as stored)
 *   W      [N][K] with gate and up rows interleaved in groups of 16: rows
 *          16b .. 16b+7 are the gate rows and rows 16b+8 .. 16b+15 the up rows
 *          of outputs 8b .. 8b+7.  N % 16 == 0 (else DL_ERR_UNSUPPORTED_SHAPE).
 *   bias   bf16 [N] in the same row order, or NULL
 *   y      bf16 [M][N/2]; y_f32 fp32 [M][N/2] or NULL (the value before rounding)
 *   everything else as for dl_linear_bf16 / dl_linear_fp8_block128, with the
 *   same workspace (dl_workspace_bytes(M, N, K, dtype)).
 */
dl_status dl_linear_swiglu(int dtype, const void* x, const void* W, const float* scales,
                           const void* bias, void* y, float* y_f32, int M, int N, int K,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * A linear layer (typically the lm_head) with the greedy-decoding argmax fused
 * into its epilogue: for every row m,
 *     idx[m] = the lowest n among the largest y[m][n] (+ bias),
 * decided on the fp32 values before rounding; a NaN counts as larger than any
 * number (the first NaN wins) and -0 equals +0.  This is the on-device argmax
 * of "Developing a custom Qwen2.5 72B inference engine from scratch", §5 (pick
 * the next token on the GPU instead of copying the logits to the host), fused
 * into the last linear of the step: the logits need not be written at all.
 *   dtype, x, W, scales, bias, M, N, K, workspace, ws_bytes, stream:
 *          as for dl_linear_bf16 / dl_linear_fp8_block128
 *   idx    int32 [M] (required, 4-byte aligned)
 *   maxval fp32 [M] or NULL: the largest value itself
 *   y      bf16 [M][N] or NULL; y_f32 fp32 [M][N] or NULL: the logits, if wanted
 * Every candidate is reduced to a 64-bit key whose maximum does not depend on
 * the order of combination, so the result is exact and reproducible.
 */
dl_status dl_linear_argmax(int dtype, const void* x, const void* W, const float* scales,
                           const void* bias, int* idx, float* maxval, void* y, float* y_f32, int M,
                           int N, int K, void* workspace, size_t ws_bytes, void* stream);

/* One layer of a decode weight stream (see dl_decode_stream). */
typedef struct dl_layer {
    int dtype;             /* dl_dtype                                    */
    int M, N, K;
    const void* x;         /* bf16 [M][K]                                 */
    const void* W;         /* bf16 [N][K] or e4m3 codes [N][K]            */
    const float* scales;   /* FP8 only: fp32 [ceil(N/128)][K/128]; else NULL */
    const void* bias;      /* bf16 [N] or NULL                            */
    void* y;               /* bf16 [M][N]; [M][N/2] with act = 1; int32 [M] with act = 2 */
    int act;               /* 0: plain; 1: SwiGLU (as dl_linear_swiglu);
                              2: argmax (as dl_linear_argmax: y receives the indices,
                              no logits are written)                      */
} dl_layer;

/*
 * Run layers[0..n_layers) back to back on one stream, in order, with no host
 * synchronisation between them -- the whole weight stream of a decode step
 * (e.g. 80 x {QKV, O, gate_up, down} + lm_head).  A layer may read the y of
 * an earlier layer as its x.  All layers are validated before anything is
 * enqueued.  ws_bytes must cover the largest layer.
 * use_graph = 1: the sequence is captured once into a CUDA graph, cached
 * under the exact contents of `layers` (pointers, shapes) + workspace, and
 * replayed on later calls with the same list, removing per-launch host cost
 * (a decode step replayed on the GPU with no host involvement; engine page §5).
 * The first call with a new list captures on `stream`, which therefore must
 * not itself be capturing.  dl_graph_cache_clear() drops cached graphs.
 */
dl_status dl_decode_stream(const dl_layer* layers, int n_layers, void* workspace,
                           size_t ws_bytes, void* stream, int use_graph);

/*
 * Workspace bytes with which dl_decode_stream makes every FP8 layer's exact
 * f16 activation copy without a prep launch of its own where it can:
 *  - made ahead: an FP8 layer whose x no earlier layer of the list writes (no
 *    byte of its x lies in an earlier layer's y): layer 0's copy just before
 *    it, the others in batches, one launch right after every 16th layer
 *    (layer 16k) holding the copies of layers 16k+1 .. 16k+16 and running
 *    alongside layer 16k (the first batch before layer 0 if layer 0 is not
 *    such a layer); one region per such layer;
 *  - made by the layer before: an FP8 layer whose x is exactly the whole y of
 *    the layer just before it, a plain linear (act 0) with the same M (and so
 *    N % 128 == 0): that layer's epilogue writes the copy next to y; two
 *    alternating regions and per-CTA slots for those producers.
 * Plus the largest layer's dl_workspace_bytes.  With a smaller workspace (at
 * least the largest layer's) the call is still correct, with the same
 * results bit for bit: layers whose copy does not fit get a prep launch.  0
 * if the list is invalid.  Host-only apart from reading device attributes.
 */
size_t dl_decode_stream_workspace_bytes(const dl_layer* layers, int n_layers);

/*
 * Kernel launches one dl_decode_stream call over this list enqueues with a
 * workspace of ws_bytes (prep launches included), or -1 if the list is
 * invalid.  Host-only apart from reading device attributes.
 */
int dl_decode_stream_launches(const dl_layer* layers, int n_layers, size_t ws_bytes);

/*
 * Destroy every cached graph (host call; synchronises nothing: a graph still
 * running is freed once its launches complete).  The cache keeps at most 16
 * graphs and drops the least recently used one when a new list is captured.
 */
void dl_graph_cache_clear(void);

/* Number of graphs currently cached by dl_decode_stream (host call). */
int dl_graph_cache_size(void);

/*
 * Process-wide tuning overrides, for tests and tuning; 0 = automatic.
 *   kernel       dl_kernel family to force
 *   ctas_per_sm  resident CTAs per SM the persistent grid is sized for: 1
 *                (one CTA with all of the SM's shared memory) or 2 (two, half
 *                each); 0 = 1
 *   max_ctas     upper bound on the grid (1 = a single CTA)
 * Changing an override changes dl_workspace_bytes and may change the last
 * bits of results (a different split of K); any setting is correct.
 * ctas_per_sm = 2 is not applied to FP8 calls with more than 8 tokens (16
 * staged token rows): they keep one CTA per SM.
 * Not thread-safe against concurrent launches.
 */
dl_status dl_set_override(int kernel, int ctas_per_sm, int max_ctas);

/*
 * Test hooks for the bounded device waits, applied to later launches
 * (process-wide, like the overrides; 0, 0 restores normal operation):
 *   wait_limit_ns   how long every device-side wait waits before it gives up,
 *                   sets its bit of the device error word and lets its CTA
 *                   leave (0 = the default, about 2 s);
 *   withhold_stage  k >= 1: CTA 0 of every later linear-layer launch opens its
 *                   k-th pipeline stage (the stage's barrier expects its
 *                   bytes) but never issues the copies that would fill it, so
 *                   every wait on that stage runs out; no copy is in flight
 *                   for it when the CTA leaves.  Needs 0 < wait_limit_ns <=
 *                   100 ms (else DL_ERR_INVALID_ARG).
 * A launch that ran with a withheld stage leaves wrong outputs and may leave
 * arrival counters set in its workspace: zero the workspace's first
 * DL_WORKSPACE_ZERO_BYTES before using it again, and read the error word with
 * dl_device_status.  Not thread-safe against concurrent launches.
 */
dl_status dl_set_wait_test(long long wait_limit_ns, int withhold_stage);

/*
 * Read and clear the device error word of the current device: bit 0 = a
 * consumer gave up waiting for a weight tile, bit 1 = the loader gave up
 * waiting for a free stage, bit 2 = the final wait for copies in flight gave
 * up, bit 3 = a hand-over of a split-K run between the consumer warps and the
 * ticket warp gave up.  Every device wait is bounded (about 2 s, or the limit
 * set with dl_set_wait_test); a kernel that gives up sets a bit and returns
 * instead of hanging.  SYNCHRONISES the device.  *flags may
 * be NULL.  Returns DL_ERR_DEVICE if any bit was set.
 */
dl_status dl_device_status(unsigned int* flags);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* dl_last_error(void);

/* DL_VERSION of the loaded library. */
int dl_version(void);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* DL_LINEAR_H */
