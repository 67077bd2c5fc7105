// The decode-linear kernel: y[M,N] = x[M,K] . w[N,K]^T (+ bias), M <= 16.
//
// Work decomposition.  The weight matrix is cut into tiles of kBN = 128 rows;
// each tile's K range is cut into units of 32 KB of weights: 128 columns of
// bf16, or 256 columns (two 128x128 scale blocks) of FP8.  The U = tiles x
// units-per-tile units, in tile-major order, are cut into
// contiguous segments by a partition fixed by (dtype, M, N, K, SM count)
// alone.  A persistent grid of about one CTA per SM takes segment blockIdx.x
// of the first wave.  For FP8, and for bf16 layers of at most 128 units per
// CTA, that wave is the whole partition: a static balanced split, every CTA
// within one unit of the others.  For larger bf16 layers the first wave holds
// about 7/8 of the work and waves of segments that halve in size down to a
// small minimum follow; CTAs claim those in order from an atomic counter, so
// SMs that happen to stream faster take more of the small segments and all of
// them finish together.  Either way the long dimension is
// spread over blocks so that every SM streams weights, as in "9% faster
// GLM-5.3-Flash prefill with GPU-to-GPU IPC" (section "TileLang: twice as
// fast, and no faster", where a 1..6-token step otherwise launches 16-96
// blocks for 188 SMs).
//
// Pipeline.  Warp 8 (one elected thread) streams units HBM -> shared memory
// with TMA tensor copies into a ring of `stages` buffers guarded by full/empty
// mbarriers; each buffer carries a header naming its unit (and, for FP8, the
// unit's block scale and the per-token unscale factors of its activations,
// copied asynchronously on the same barrier).  The weight tile is copied as
// 128 rows x 128 bytes with the 128-byte swizzle.  Warps 0-7 each own 16
// weight rows of the tile (the TileLang loop's two-stage software pipeline,
// deepened to cover GB300's HBM latency).  Every weight byte is read from HBM
// exactly once per call.
//
// FP8 activations.  Before the main kernel, a prep kernel (dl_kernels_fp8.cu)
// writes a copy of x in f16, each (token, 128-column block) scaled by a power of two chosen so
// that the copy is exact, and the power of two that undoes it (0 when no such
// power exists).  e4m3 codes convert exactly to f16 in one hardware
// instruction per pair, so FP8 units multiply f16 weights by f16 activations
// with fp32 accumulation, and the unscale factor and the block scale are
// applied to each block's fp32 partial.  A unit whose activations are not
// exact in f16 (rare: a block spanning more than ~32 binades, or inf/NaN)
// runs the same products from the bf16 x in global memory with an exact
// e4m3 -> bf16 decode.
//
// Consumer families:
//   SIMT: one weight row per lane (two lanes per row, one per K half), CUDA-core
//         mixed-precision fused multiply-adds (bf16 x bf16 or f16 x f16 ->
//         fp32; the row-tiled GEMV of "Developing a custom Qwen2.5 72B
//         inference engine from scratch", §6.1); a shuffle joins the two
//         halves at the end of a run.
//   MMA:  warp-level mma.sync m16n8k16 -> fp32 with the weights as the 16-row A
//         operand and the (<= 16) tokens as the B operand (the
//         16-bit GEMM of the TileLang loop, activations against the
//         dequantised weight tile with the weights' rows as columns), in
//         bf16 for bf16 weights and in f16 for FP8 weights.
//   TC:   (FP8, opt-in) 5th-generation tensor cores: an MMA warp issues
//         tcgen05.mma kind::f8f6f4 with the e4m3 weight tile, as TMA wrote it,
//         as the A operand and an exact three-part e4m3 split of x as B; the
//         fp32 accumulators live in tensor memory and warps 0-3 read them back.
//         Correct and tested, but slower here than MMA (a stage is released
//         only once the tensor core has read it).
// SIMT and MMA keep two accumulator sets alternating over the K steps
// (shorter dependency chains), added in a fixed order.
//
// Split-K fix-up.  Within one segment the units of one tile form a "run".  A
// run that covers its whole tile is finished on the spot: every warp rounds
// its own rows (+ bias) to bf16 and stores them.  Otherwise the warps store
// their fp32 partial rows in the workspace slot of the run's (segment,
// first-or-last tile) pair and arrive on a barrier; a ticket warp (warp 9)
// waits for all eight, then takes the tile's arrival ticket with an
// acquire-release atomic -- the memory fence it implies stalls only that warp
// -- and publishes whether this was the last contribution.  The consumers read
// that result at their next split run end (or exit), long after it is ready;
// if the tile is complete, all of them sum its slots in segment order (=
// ascending K), add the bias, round once and reset the ticket.  No CTA ever waits for another, and the order of every sum is fixed
// by the partition alone, so results are bitwise reproducible whichever CTA
// computed which segment.  Inside one GPU this plays the role of the
// row-parallel split of "Multi-GPU Inference and Serving at Scale", Example 3,
// whose partial sums an all-reduce adds.
//
// Dependent launch.  The kernel lets the next kernel on the stream launch as
// soon as it starts (griddepcontrol.launch_dependents); all its threads but
// the loader sleep in griddepcontrol.wait until the previous kernel has
// finished, and the loader touches nothing that kernel may have written before
// that wait -- except, when `early_stages` is set (the kernels before it are
// known never to write weights or scales: earlier layers of one
// dl_decode_stream call, or for a single FP8 call the activation prep kernel,
// which waits for its own predecessor before it lets this one launch), the
// weight tiles and scales of its first stages, which it prefetches meanwhile.
//
// Every wait is bounded (mbarrier waits give up after ~2 s, set a bit of the
// device error word and make the CTA leave in an orderly way).
//
// Next-layer activation copy.  Inside one decode stream, a plain linear whose
// y is exactly the x of a following FP8 layer also writes that layer's exact
// f16 copy (xh_next): every output tile is one 128-column K block of it, made
// by the fix-up (one warp per token) next to y; tiles one segment covers whole
// go through per-CTA slots and a bounded meeting of the consumer warps.
#pragma once

#include "dl_device.cuh"

namespace dl {

constexpr int kBN = 128;                 // weight rows per tile
constexpr int kBK = 128;                 // K columns per unit (one FP8 scale block)
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kLoaderWarp = kConsumerWarps;       // warp 8: TMA producer
constexpr int kTicketWarp = kConsumerWarps + 1;   // warp 9: split-K arrival tickets
constexpr int kMmaWarp = kConsumerWarps + 2;      // warp 10 (tensor-memory family): MMA issue
constexpr int kThreads = kConsumerThreads + 64;
constexpr int kMaxWaves = 24;
constexpr int kUnscaleStride = 16;       // unscale factors per k-block (one per token slot)
// The most stages a loader may have in flight when it claims another segment:
// enough to cover HBM latency at one SM's share of the bandwidth, few enough
// that the last claims leave little backlog.
constexpr int kClaimDepth = 3;

enum DType { kBF16 = 0, kFP8 = 1 };
enum Family { kSIMT = 1, kMMA = 2, kTC = 3 };

// Tensor-memory family (FP8 only): B-operand rows per K block (3 activation
// parts x the token slots), the MMA's N (a multiple of 16; MT = 8 reads 8
// rows past a unit's 24, whose columns are ignored), and TMEM columns: two
// buffers of two units.
template <int MT>
struct TcShape {
    static constexpr int rows = 3 * MT;
    static constexpr int n = rows < 32 ? 32 : rows;
    static constexpr int cols = 2 * 2 * n <= 128 ? 128 : 256;
};

// Stage header flags.
constexpr int kRunFirst = 1;   // first unit of a run (a run = one tile inside one segment)
constexpr int kRunLast = 2;    // last unit of a run
constexpr int kDone = 4;       // no more work: consumers leave

struct LinearParams {
    const uint16_t* bias;     // bf16 [N] or null
    uint16_t* y;              // bf16 [M][N]
    float* y_f32;             // fp32 [M][N] or null
    const float* scales;      // fp32 [ceil(N/128)][KB] (FP8)
    int scale_off;            // FP8: elements between the scales tensor map's base (the
                              //   scales rounded down to 16 bytes) and scales[0] (0..3)
    const uint16_t* x;        // bf16 [M][K] (FP8: read only by units not exact in f16)
    const float* unscale;     // fp32 [KB][16] (FP8): 2^-s of the f16 copy, 0 = not exact
    int* counter;             // [0]: segments claimed after the first wave, [1]: CTAs done
                              //   claiming, [2]: consumer warps finished (argmax)
    unsigned long long* best; // argmax: [16] best key per token (in the zero prefix)
    int* idx;                 // argmax: int32 [M] result
    float* maxval;            // argmax: fp32 [M] largest logit, or null
    int* tickets;             // [n_tiles] arrival counters (zero between calls)
    float* partials;          // [n_segments][2][MTB][kBN] fp32 (scratch)
    int M, N, K;
    int act;                  // 0: y = x.W^T (+ bias); 1: SwiGLU over gate/up row pairs;
                              //   2: also the argmax over n of every row m (see below)
    int ny;                   // row stride of y (N, or N / 2 with SwiGLU)
    int KB;                   // 128-column K blocks per tile = ceil(K / 128)
    int UT;                   // partition units per tile: bf16 one K block each (UT = KB),
                              //   FP8 two (UT = ceil(KB / 2), the last one single if KB is odd)
    int n_tiles;
    long long units;          // n_tiles * UT
    int n_segments;
    int n_waves;              // the partition: wave w holds segments
    int wave_seg0[kMaxWaves + 1];     //   [wave_seg0[w], wave_seg0[w+1]), each of
    long long wave_unit0[kMaxWaves];  //   wave_size[w] units from wave_unit0[w]
    int wave_size[kMaxWaves];         //   (the very last segment ends at U)
    int stages;
    int early_stages;         // stages whose weights may be fetched before griddepcontrol.wait
                              //   (0: the previous kernel may write weights)
    unsigned* err;            // device error word (bounded waits OR their bit in)
    unsigned long long wait_ns;   // how long a device wait waits before it gives up
    int withhold;             // test hook: k >= 1 = CTA 0 opens its k-th stage but never
                              //   issues the copies that fill it (0: off)
    // The exact f16 copy of y for a next FP8 layer whose x is this layer's y
    // (act 0, N % 128 == 0; its copy has the same staged token rows MTB):
    // xh_next [N/128][2][MTB][64] and us_next [N/128][16], written by the
    // epilogue of every tile (tile t = K block t of the next layer), or null.
    uint16_t* xh_next;
    float* us_next;
    float* wslot;             // with xh_next: [gridDim.x][2][MTB][kBN] fp32, a CTA's
                              //   slots for the tiles one segment covers whole
};

// One pipeline stage holds one unit, or for FP8 up to two consecutive units
// of one run (the same 32 KB of weights as a bf16 unit).
constexpr int kMaxUnitsPerStage = 2;

struct StageHeader {
    // FP8: one tensor copy of 8 block scales (32 bytes; a tensor copy lands
    // on a 128-byte boundary, so the header is 256 bytes and the box comes
    // first): the scale of K block kb is scale8[soff], of kb + 1 scale8[soff + 1]
    float scale8[8];
    int tile;                 // units held by the stage: weight rows 128*tile..,
    int kb;                   //   K blocks kb .. kb + nkb - 1
    int seg;                  // segment they belong to
    int flags;                // kRunFirst | kRunLast | kDone
    int nkb;                  // units in the stage (1, or 2 for FP8)
    int soff;                 // FP8: position of K block kb's scale in scale8 (0..3)
    int pad[2];
    float unscale[kMaxUnitsPerStage][kUnscaleStride];   // FP8: per-token unscale factors
    int pad2[16];
};
static_assert(sizeof(StageHeader) == 256, "stage header layout");

template <int DT>
struct TileBytes {
    static constexpr int w = kBN * kBK * (DT == kBF16 ? 2 : 1);   // one unit
};
constexpr int kStageWBytes = 2 * kBN * kBK;   // weights of one stage (either dtype)

template <int MT>
struct XRows {
    static constexpr int v = MT < 8 ? 8 : MT;   // token rows staged (zero-filled past M)
};

// Shared-memory layout of one CTA (offsets from a 1024-aligned base).  The
// host sizes the launch with the same function.
struct SmemLayout {
    int w, x, hdr, bars, runs, best, total;
};

// Hand-over of one split run between the consumer warps and the ticket warp
// (two slots, used alternately).
struct RunSlot {
    int tile;                 // tile of the run (-1: no more runs)
    int jf, jl;               // first and last segment contributing to the tile
    int last;                 // ticket result: tile if this run completed it, else -1
};

__host__ __device__ constexpr SmemLayout smem_layout(int dtype, int family, int mt, int stages) {
    const int mtb = mt < 8 ? 8 : mt;
    const int wbytes = kStageWBytes;
    const int xbytes = family == kTC ? kMaxUnitsPerStage * 3 * mtb * 128
                                     : mtb * kBK * 2 * (dtype == kBF16 ? 1 : kMaxUnitsPerStage);
    SmemLayout L{};
    L.w = 0;
    L.x = L.w + stages * wbytes;
    L.hdr = L.x + stages * xbytes;
    L.bars = L.hdr + stages * (int)sizeof(StageHeader);
    // full[S], empty[S], written[2], result[2], xch, mma_done[2], tmem_free[2],
    // the TMEM address (8 bytes)
    L.runs = L.bars + (2 * stages + 10) * 8;
    L.best = L.runs + 2 * (int)sizeof(RunSlot) + 16;      // [8 warps][16 tokens] argmax keys
    L.total = L.best + kConsumerWarps * 16 * 8;
    return L;
}

// Threads of a CTA: 8 consumer warps, the loader warp and the ticket warp
// (and the MMA-issue warp of the tensor-memory family).
__host__ __device__ constexpr int threads_for(int, int family) {
    return family == kTC ? kThreads + 32 : kThreads;
}

// CTAs per SM an instance is compiled for: one, with the whole register file
// and shared memory of the SM.  (A grid of two CTAs per SM can still be asked
// for; they are then co-resident only where the registers allow it.)
__host__ __device__ constexpr int min_blocks_for(int, int, int) { return 1; }

// First unit of segment j (j = n_segments gives U).
__device__ __forceinline__ long long seg_begin(const LinearParams& p, int j) {
    if (j >= p.n_segments) return p.units;
    int w = 0;
    while (w + 1 < p.n_waves && p.wave_seg0[w + 1] <= j) ++w;
    const long long u = p.wave_unit0[w] + (long long)(j - p.wave_seg0[w]) * p.wave_size[w];
    return u < p.units ? u : p.units;
}

// Segment holding unit u (0 <= u < U).
__device__ __forceinline__ int seg_of(const LinearParams& p, long long u) {
    int w = 0;
    while (w + 1 < p.n_waves && p.wave_unit0[w + 1] <= u) ++w;
    return p.wave_seg0[w] + (int)((u - p.wave_unit0[w]) / p.wave_size[w]);
}

// ------------------------------------------------------------------ epilogue

// Final value (+ bias) of output (m, n), stored to y / y_f32 where given; the
// value is returned for the argmax epilogue.
__device__ __forceinline__ float write_output(const LinearParams& p, int m, int n, float v) {
    if (p.bias) v += bf16_bits_to_f32(p.bias[n]);
    const long long o = (long long)m * p.ny + n;
    if (p.y) p.y[o] = f32_to_bf16_rne(v);
    if (p.y_f32) p.y_f32[o] = v;
    return v;
}

// Argmax epilogue (act = 2).  A candidate (value v, index n) becomes one 64-bit
// key whose unsigned order is the selection order: the high word orders the
// floats (NaN above everything, -0 equal to +0), the low word is 2^32-1-n so
// that among equal values the lowest index wins.  The maximum over keys does
// not depend on the order candidates are combined in: results are exact and
// reproducible.  0 is below every candidate.
__device__ __forceinline__ unsigned long long argmax_key(float v, int n) {
    v += 0.f;                                            // -0 -> +0
    const unsigned b = __float_as_uint(v);
    const unsigned o = (v != v) ? 0xffffffffu : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
    return ((unsigned long long)o << 32) | (0xffffffffu - (unsigned)n);
}

__device__ __forceinline__ float argmax_key_value(unsigned long long k) {
    const unsigned o = (unsigned)(k >> 32);
    if (o == 0xffffffffu) return __uint_as_float(0x7fffffffu);      // NaN
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ unsigned long long max_u64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

// Largest key among the lanes of `mask` reached by the xor offsets >= `from`.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k, int from) {
#pragma unroll
    for (int o = 16; o >= from; o >>= 1) k = max_u64(k, __shfl_xor_sync(0xffffffffu, k, o));
    return k;
}

// SwiGLU epilogue.  The weight rows come in groups of 16: rows 16b .. 16b + 7
// are the gate rows and rows 16b + 8 .. 16b + 15 the up rows of outputs 8b ..
// 8b + 7.  With g and u the full fp32 sums (+ bias) of a pair,
// y[m][j] = silu(g) * u = g / (1 + e^-g) * u, rounded once to bf16.  `ng` is
// the gate row, j = 8 (ng / 16) + ng % 16 the output column.
__device__ __forceinline__ void write_swiglu(const LinearParams& p, int m, int ng, float g, float u) {
    if (p.bias) {
        g += bf16_bits_to_f32(p.bias[ng]);
        u += bf16_bits_to_f32(p.bias[ng + 8]);
    }
    const float v = g / (1.f + expf(-g)) * u;
    const long long o = (long long)m * p.ny + (ng >> 4) * 8 + (ng & 15);
    p.y[o] = f32_to_bf16_rne(v);
    if (p.y_f32) p.y_f32[o] = v;
}

// Store one finished value of a run: to y (a run that covers its whole tile,
// slot == null) or to the run's partial slot [MTB][kBN] (row within the tile).
__device__ __forceinline__ void put_value(const LinearParams& p, float* slot, int n0, int m,
                                          int row, float v) {
    if (m >= p.M) return;
    if (slot)
        slot[m * kBN + row] = v;
    else if (n0 + row < p.N)
        write_output(p, m, n0 + row, v);
}

// ------------------------------------------------------------------ consumers

// SIMT consumer.  Lane l of warp w owns weight row 16w + (l & 15) and the K
// half (l >> 4) of every unit: 64 columns = 8 chunks of 16 bytes (bf16) or 4
// chunks (fp8, 16 codes each).  acc[2][m] are the lane's two fp32 sums for
// token m (even and odd chunks).
template <int DT, int MT>
struct SimtConsumer {
    static constexpr int MTB = XRows<MT>::v;
    float acc[2][MT];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[0][m] = acc[1][m] = 0.f;
    }

    // sw: weight tile of the unit; sx: its activations (bf16, or for FP8 the
    // exact f16 copy); FP8: its block scale, the per-token unscale factors and
    // its K block.
    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, float scale,
                                            const float* unscale, int kb, const LinearParams& p,
                                            int warp, int lane) {
        const int row = warp * 16 + (lane & 15);
        const int h = lane >> 4;
        const int sw8 = row & 7;
        const uint32_t xbase = sx + h * (MTB * 128);
        if constexpr (DT == kBF16) {
            const uint32_t wbase = sw + h * (kBN * 128) + row * 128;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 w = lds128(wbase + ((cc ^ sw8) << 4));
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    const uint4 xv = lds128(xbase + m * 128 + ((cc ^ (m & 7)) << 4));
                    float a = acc[cc & 1][m];
                    a = fma2_bf16(w.x, xv.x, a);
                    a = fma2_bf16(w.y, xv.y, a);
                    a = fma2_bf16(w.z, xv.z, a);
                    a = fma2_bf16(w.w, xv.w, a);
                    acc[cc & 1][m] = a;
                }
            }
        } else {
            float u[MT];
            bool exact = true;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                u[m] = unscale[m];
                exact &= (u[m] != 0.f);      // token slots >= M carry 1
            }
            float part[2][MT];
            if (exact) {
                fp8_unit_f16(sw, xbase, row, h, sw8, part);
            } else {
                fp8_unit_exact(sw, p, kb, row, h, sw8, part);
#pragma unroll
                for (int m = 0; m < MT; ++m) u[m] = 1.f;
            }
#pragma unroll
            for (int m = 0; m < MT; ++m)
                acc[0][m] = fmaf((part[0][m] + part[1][m]) * u[m], scale, acc[0][m]);
        }
    }

    // One FP8 unit against the exact f16 copy of x: codes 16cc..16cc+15 of the
    // row (cc = 4h + j) pair with 16-column group j of x box h, stored in the
    // fragment order of the prep kernel: its word w < 4 holds columns 4w, 4w+1
    // and word 4 + w columns 4w + 2, 4w + 3.
    __device__ __forceinline__ void fp8_unit_f16(uint32_t sw, uint32_t xbase, int row, int h,
                                                 int sw8, float (&part)[2][MT]) {
        const uint32_t wbase = sw + row * 128;
#pragma unroll
        for (int m = 0; m < MT; ++m) part[0][m] = part[1][m] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cc = 4 * h + j;
            const uint4 w = lds128(wbase + ((cc ^ sw8) << 4));
            uint32_t wh[8];
            e4m3x4_to_f16x2x2(w.x, wh[0], wh[1]);
            e4m3x4_to_f16x2x2(w.y, wh[2], wh[3]);
            e4m3x4_to_f16x2x2(w.z, wh[4], wh[5]);
            e4m3x4_to_f16x2x2(w.w, wh[6], wh[7]);
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 x0 = lds128(xbase + m * 128 + (((2 * j) ^ (m & 7)) << 4));
                const uint4 x1 = lds128(xbase + m * 128 + (((2 * j + 1) ^ (m & 7)) << 4));
                float a = part[j & 1][m];
                a = fma2_f16(wh[0], x0.x, a);     // columns 0, 1
                a = fma2_f16(wh[1], x1.x, a);     //         2, 3
                a = fma2_f16(wh[2], x0.y, a);     //         4, 5
                a = fma2_f16(wh[3], x1.y, a);
                a = fma2_f16(wh[4], x0.z, a);
                a = fma2_f16(wh[5], x1.z, a);
                a = fma2_f16(wh[6], x0.w, a);
                a = fma2_f16(wh[7], x1.w, a);
                part[j & 1][m] = a;
            }
        }
    }

    // The same unit from the bf16 x in global memory with the exact e4m3 ->
    // bf16 decode (NaN codes stay NaN), for activations not exact in f16.
    __device__ __forceinline__ void fp8_unit_exact(uint32_t sw, const LinearParams& p, int kb,
                                                   int row, int h, int sw8, float (&part)[2][MT]) {
        const uint32_t wbase = sw + row * 128;
        const uint16_t* xk = p.x + (long long)kb * kBK + 64 * h;
#pragma unroll
        for (int m = 0; m < MT; ++m) part[0][m] = part[1][m] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cc = 4 * h + j;
            const uint4 w = lds128(wbase + ((cc ^ sw8) << 4));
            const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
            uint32_t wb[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wb[2 * i] = e4m3x2_to_bf16x2(wq[i] & 0xffffu);
                wb[2 * i + 1] = e4m3x2_to_bf16x2(wq[i] >> 16);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= p.M) continue;
                const uint16_t* xm = xk + (long long)m * p.K + 16 * j;
                const uint4 x0 = ldg128(xm);
                const uint4 x1 = ldg128(xm + 8);
                float a = part[j & 1][m];
                a = fma2_bf16(wb[0], x0.x, a);
                a = fma2_bf16(wb[1], x0.y, a);
                a = fma2_bf16(wb[2], x0.z, a);
                a = fma2_bf16(wb[3], x0.w, a);
                a = fma2_bf16(wb[4], x1.x, a);
                a = fma2_bf16(wb[5], x1.y, a);
                a = fma2_bf16(wb[6], x1.z, a);
                a = fma2_bf16(wb[7], x1.w, a);
                part[j & 1][m] = a;
            }
        }
    }

    // Finish a run: join the accumulators and the two K halves, store the rows
    // (SwiGLU on a finished tile: lane l < 8 pairs gate row l with up row l + 8;
    // argmax: the warp's best candidate per token goes to its row sbest[16]).
    __device__ __forceinline__ void write_rows(const LinearParams& p, float* slot, int n0, int warp,
                                               int lane, unsigned long long* sbest) {
        const int row = warp * 16 + (lane & 15);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float mine = acc[0][m] + acc[1][m];
            const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
            const float v = mine + other;
            if (p.act == 1 && !slot) {
                const float up = __shfl_xor_sync(0xffffffffu, v, 8);
                if (lane < 8 && m < p.M && n0 + row < p.N) write_swiglu(p, m, n0 + row, v, up);
            } else if (p.act == 2 && !slot) {
                unsigned long long k = 0;
                if (lane < 16 && m < p.M && n0 + row < p.N)
                    k = argmax_key(write_output(p, m, n0 + row, v), n0 + row);
                k = warp_max_key(k, 1);
                if (lane == 0 && m < p.M) sbest[m] = max_u64(sbest[m], k);
            } else if (lane < 16) {
                put_value(p, slot, n0, m, row, v);
            }
        }
    }
};

// MMA consumer.  Warp w owns rows 16w..16w+15 as the A operand of
// mma.m16n8k16; the tokens are the B operand (n = 8, two n-tiles for MT = 16).
// acc[set][nt][i] follows the mma accumulator layout: thread (g = lane/4,
// t = lane%4) holds rows g and g+8, tokens 8nt + 2t and 8nt + 2t + 1.
template <int DT, int MT>
struct MmaConsumer {
    static_assert(MT == 8 || MT == 16, "MMA consumer stages 8 or 16 tokens");
    static constexpr int NT = MT / 8;
    float acc[2][NT][4];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[k][nt][i] = 0.f;
    }

    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, float scale,
                                            const float* unscale, int kb, const LinearParams& p,
                                            int warp, int lane) {
        const int mat = lane >> 3, rr = lane & 7;
        const int arow = warp * 16 + rr + ((mat & 1) << 3);
        const int aswz = arow & 7;
        const uint32_t abase = sw + arow * 128;
        if constexpr (DT == kBF16) {
            // 8 k16 steps; step s reads bf16 chunks 2(s%4), 2(s%4)+1 of box s/4;
            // steps s (even) and s+1 go to accumulator sets 0 and 1.
#pragma unroll
            for (int s = 0; s < 8; s += 2) {
                const int box = s >> 2;
                const int c0 = (s & 3) * 2;
                uint32_t a0[4], a1[4];
                ldmatrix_x4(abase + box * (kBN * 128) + (((c0 + (mat >> 1)) ^ aswz) << 4),
                            a0[0], a0[1], a0[2], a0[3]);
                ldmatrix_x4(abase + box * (kBN * 128) + (((c0 + 2 + (mat >> 1)) ^ aswz) << 4),
                            a1[0], a1[1], a1[2], a1[3]);
                const uint32_t xbox = sx + box * (MT * 128);
                if constexpr (MT == 8) {
                    uint32_t b[4];
                    ldmatrix_x4(xbox + rr * 128 + (((c0 + mat) ^ rr) << 4), b[0], b[1], b[2], b[3]);
                    mma_bf16_16816(acc[0][0], a0[0], a0[1], a0[2], a0[3], b[0], b[1]);
                    mma_bf16_16816(acc[1][0], a1[0], a1[1], a1[2], a1[3], b[2], b[3]);
                } else {
                    const int tok = rr + ((mat >> 1) << 3);
                    uint32_t b[4], c[4];
                    ldmatrix_x4(xbox + tok * 128 + (((c0 + (mat & 1)) ^ (tok & 7)) << 4),
                                b[0], b[1], b[2], b[3]);
                    ldmatrix_x4(xbox + tok * 128 + (((c0 + 2 + (mat & 1)) ^ (tok & 7)) << 4),
                                c[0], c[1], c[2], c[3]);
                    mma_bf16_16816(acc[0][0], a0[0], a0[1], a0[2], a0[3], b[0], b[1]);
                    mma_bf16_16816(acc[0][1], a0[0], a0[1], a0[2], a0[3], b[2], b[3]);
                    mma_bf16_16816(acc[1][0], a1[0], a1[1], a1[2], a1[3], c[0], c[1]);
                    mma_bf16_16816(acc[1][1], a1[0], a1[1], a1[2], a1[3], c[2], c[3]);
                }
            }
        } else {
            const int t = lane & 3;
            float part[2][NT][4];
            float u0[NT], u1[NT];
            bool exact = true;
            if constexpr (NT == 1) {
                // 8 staged tokens: the f16 route runs first, speculatively.
                // The unit's activations are almost always exact in f16, and
                // deciding first would put the unscale loads and the warp vote
                // in front of every MMA (same-box: FP8 M = 6 layer step
                // -0.7 %).  A unit that is not exact is recomputed on the exact
                // route and the f16 sums are discarded, so the results are
                // those of deciding first.
                fp8_unit_f16(abase, aswz, mat, sx, lane, part);
                u0[0] = unscale[2 * t];
                u1[0] = unscale[2 * t + 1];
                exact = (u0[0] != 0.f) && (u1[0] != 0.f);      // token slots >= M carry 1
                if (!__all_sync(0xffffffffu, exact)) {
                    fp8_unit_exact(abase, aswz, mat, p, kb, lane, part);
                    u0[0] = u1[0] = 1.f;
                }
            } else {
                // 16 tokens (twice the fragments in flight): deciding first
                // measured faster.
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    u0[nt] = unscale[8 * nt + 2 * t];
                    u1[nt] = unscale[8 * nt + 2 * t + 1];
                    exact &= (u0[nt] != 0.f) && (u1[nt] != 0.f);   // token slots >= M carry 1
                }
                if (__all_sync(0xffffffffu, exact)) {
                    fp8_unit_f16(abase, aswz, mat, sx, lane, part);
                } else {
                    fp8_unit_exact(abase, aswz, mat, p, kb, lane, part);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) u0[nt] = u1[nt] = 1.f;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                acc[0][nt][0] = fmaf((part[0][nt][0] + part[1][nt][0]) * u0[nt], scale, acc[0][nt][0]);
                acc[0][nt][1] = fmaf((part[0][nt][1] + part[1][nt][1]) * u1[nt], scale, acc[0][nt][1]);
                acc[0][nt][2] = fmaf((part[0][nt][2] + part[1][nt][2]) * u0[nt], scale, acc[0][nt][2]);
                acc[0][nt][3] = fmaf((part[0][nt][3] + part[1][nt][3]) * u1[nt], scale, acc[0][nt][3]);
            }
        }
    }

    // Fragments of k-steps s and s + 1: the A codes of both steps and their
    // B fragments (chunks c0 .. c0 + 3 of box s / 4).
    __device__ __forceinline__ void fp8_load_pair(uint32_t abase, int aswz, int mat, uint32_t sx, int rr,
                                                  int s, uint32_t (&q)[4], uint32_t (&b)[2][NT][2]) {
        ldmatrix_x4(abase + (((s + (mat >> 1)) ^ aswz) << 4), q[0], q[1], q[2], q[3]);
        const uint32_t xbox = sx + (s >> 2) * (MT * 128);
        const int c0 = (s & 3) * 2;
        if constexpr (MT == 8) {
            uint32_t r[4];
            ldmatrix_x4(xbox + rr * 128 + (((c0 + mat) ^ rr) << 4), r[0], r[1], r[2], r[3]);
            b[0][0][0] = r[0]; b[0][0][1] = r[1];
            b[1][0][0] = r[2]; b[1][0][1] = r[3];
        } else {
            const int tok = rr + ((mat >> 1) << 3);
            uint32_t r[4], u[4];
            ldmatrix_x4(xbox + tok * 128 + (((c0 + (mat & 1)) ^ (tok & 7)) << 4), r[0], r[1], r[2], r[3]);
            ldmatrix_x4(xbox + tok * 128 + (((c0 + 2 + (mat & 1)) ^ (tok & 7)) << 4), u[0], u[1], u[2], u[3]);
            b[0][0][0] = r[0]; b[0][0][1] = r[1]; b[0][1][0] = r[2]; b[0][1][1] = r[3];
            b[1][0][0] = u[0]; b[1][0][1] = u[1]; b[1][1][0] = u[2]; b[1][1][1] = u[3];
        }
    }

    // Decode and multiply the fragments of one k-step pair.
    __device__ __forceinline__ void fp8_mma_pair(const uint32_t (&q)[4], const uint32_t (&b)[2][NT][2],
                                                 float (&part)[2][NT][4]) {
#pragma unroll
        for (int ss = 0; ss < 2; ++ss) {
            uint32_t A0, A1, A2, A3;
            e4m3x4_to_f16x2x2(q[2 * ss], A0, A2);       // row g
            e4m3x4_to_f16x2x2(q[2 * ss + 1], A1, A3);   // row g + 8
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                mma_f16_16816(part[ss][nt], A0, A1, A2, A3, b[ss][nt][0], b[ss][nt][1]);
        }
    }

    // One FP8 unit (this warp's 16 rows x 128 codes) as an f16 MMA against the
    // exact f16 copy of x.  Step s is the 16-code chunk s of each row.  Thread
    // (g, t) receives codes 4t..4t+3 of its rows' chunk; they stand for
    // fragment columns {2t, 2t+1} and {2t+8, 2t+9}, and the prep kernel stored
    // x in that order, so the B fragments come from ldmatrix exactly as for
    // bf16 weights (bank-conflict free on the swizzled tile).  The fragments of
    // the next k-step pair are loaded before the current pair's MMAs (two
    // register sets), so that their shared-memory latency overlaps the MMAs.
    __device__ __forceinline__ void fp8_unit_f16(uint32_t abase, int aswz, int mat, uint32_t sx,
                                                 int lane, float (&part)[2][NT][4]) {
        const int rr = lane & 7;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[k][nt][i] = 0.f;
        uint32_t qa[4], qb[4], ba[2][NT][2], bb[2][NT][2];
        fp8_load_pair(abase, aswz, mat, sx, rr, 0, qa, ba);
#pragma unroll
        for (int s = 0; s < 8; s += 4) {
            fp8_load_pair(abase, aswz, mat, sx, rr, s + 2, qb, bb);
            fp8_mma_pair(qa, ba, part);
            if (s + 4 < 8) fp8_load_pair(abase, aswz, mat, sx, rr, s + 4, qa, ba);
            fp8_mma_pair(qb, bb, part);
        }
    }

    // The same products as a bf16 MMA with the exact e4m3 -> bf16 decode (NaN
    // codes stay NaN) against the bf16 x in global memory, for activations
    // not exact in f16.  Same K permutation as fp8_unit_f16.
    __device__ __forceinline__ void fp8_unit_exact(uint32_t abase, int aswz, int mat,
                                                   const LinearParams& p, int kb, int lane,
                                                   float (&part)[2][NT][4]) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[k][nt][i] = 0.f;
        const uint16_t* xk = p.x + (long long)kb * kBK + 4 * t;
#pragma unroll 1
        for (int s = 0; s < 8; s += 2) {
            uint32_t q[4];
            ldmatrix_x4(abase + (((s + (mat >> 1)) ^ aswz) << 4), q[0], q[1], q[2], q[3]);
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int step = s + ss;
                const uint32_t rlo = q[2 * ss], rhi = q[2 * ss + 1];
                const uint32_t A0 = e4m3x2_to_bf16x2(rlo & 0xffffu);
                const uint32_t A2 = e4m3x2_to_bf16x2(rlo >> 16);
                const uint32_t A1 = e4m3x2_to_bf16x2(rhi & 0xffffu);
                const uint32_t A3 = e4m3x2_to_bf16x2(rhi >> 16);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = g + 8 * nt;
                    const uint2 xb = tok < p.M ? ldg64(xk + (long long)tok * p.K + 16 * step)
                                               : make_uint2(0u, 0u);
                    mma_bf16_16816(part[ss][nt], A0, A1, A2, A3, xb.x, xb.y);
                }
            }
        }
    }

    // Finish a run: add the accumulator sets and store the warp's rows
    // (SwiGLU on a finished tile: this thread holds gate row g and up row g + 8;
    // argmax: the warp's best candidate per token goes to its row sbest[16]).
    __device__ __forceinline__ void write_rows(const LinearParams& p, float* slot, int n0, int warp,
                                               int lane, unsigned long long* sbest) {
        const int g = lane >> 2, t = lane & 3;
        const int row = warp * 16 + g;
        if (p.act == 2 && !slot) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int tt = 0; tt < 2; ++tt) {
                    const int tok = 8 * nt + 2 * t + tt;
                    unsigned long long k = 0;
                    if (tok < p.M) {
                        if (n0 + row < p.N)
                            k = argmax_key(write_output(p, tok, n0 + row, acc[0][nt][tt] + acc[1][nt][tt]),
                                           n0 + row);
                        if (n0 + row + 8 < p.N)
                            k = max_u64(k, argmax_key(write_output(p, tok, n0 + row + 8,
                                                                   acc[0][nt][2 + tt] + acc[1][nt][2 + tt]),
                                                      n0 + row + 8));
                    }
                    k = warp_max_key(k, 4);              // over g: lanes with this t
                    if (g == 0 && tok < p.M) sbest[tok] = max_u64(sbest[tok], k);
                }
            return;
        }
        if (p.act == 1 && !slot) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int tok = 8 * nt + 2 * t;
                if (n0 + row >= p.N) continue;
                if (tok < p.M)
                    write_swiglu(p, tok, n0 + row, acc[0][nt][0] + acc[1][nt][0],
                                 acc[0][nt][2] + acc[1][nt][2]);
                if (tok + 1 < p.M)
                    write_swiglu(p, tok + 1, n0 + row, acc[0][nt][1] + acc[1][nt][1],
                                 acc[0][nt][3] + acc[1][nt][3]);
            }
            return;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = 8 * nt + 2 * t;
            put_value(p, slot, n0, tok, row, acc[0][nt][0] + acc[1][nt][0]);
            put_value(p, slot, n0, tok + 1, row, acc[0][nt][1] + acc[1][nt][1]);
            put_value(p, slot, n0, tok, row + 8, acc[0][nt][2] + acc[1][nt][2]);
            put_value(p, slot, n0, tok + 1, row + 8, acc[0][nt][3] + acc[1][nt][3]);
        }
    }
};

// Tensor-memory consumer (FP8, kind::f8f6f4 MMAs issued by the MMA warp).
// The MMA of a unit leaves D[row][n] in TMEM, row = weight row of the tile
// (TMEM lane), column n = part * MT + token slot.  Warps 0-3 each read the
// 32 lanes of their TMEM quadrant, so thread (w, l) owns weight row 32 w + l
// and acc[m] is its sum for token m; warps 4-7 hold nothing.
template <int MT>
struct TcConsumer {
    static_assert(MT == 8 || MT == 16, "tensor-memory consumer stages 8 or 16 tokens");
    float acc[MT];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    }

    // Add one unit's D (columns at taddr) times the unscale factors and the
    // block scale: value = (d0 + d1 2^-4) + d2 2^-8 for the three parts.
    __device__ __forceinline__ void add_tmem_unit(uint32_t taddr, const float (&u)[MT], float scale) {
        constexpr int C = TcShape<MT>::rows;          // 24 or 48 columns used
        float d[C + (C % 16 ? 16 - C % 16 : 0)];
#pragma unroll
        for (int c = 0; c < C; c += 16) {
            float v[16];
            tmem_ld16(taddr + c, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) d[c + i] = v[i];
        }
        tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float v = fmaf(d[2 * MT + m], 0.00390625f, fmaf(d[MT + m], 0.0625f, d[m]));
            acc[m] = fmaf(v * u[m], scale, acc[m]);
        }
    }

    // One unit from the bf16 x in global memory with the exact e4m3 -> bf16
    // decode (NaN codes stay NaN), for a unit whose activations the parts do
    // not hold exactly: row `row` of the 128B-swizzled weight tile at sw.
    __device__ __forceinline__ void add_exact_unit(uint32_t sw, const LinearParams& p, int kb, int row,
                                                   float scale) {
        const uint16_t* xk = p.x + (long long)kb * kBK;
        float part[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) part[m] = 0.f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
            const uint4 w = lds128(sw + row * 128 + ((c ^ (row & 7)) << 4));
            const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
            uint32_t wb[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                wb[2 * i] = e4m3x2_to_bf16x2(wq[i] & 0xffffu);
                wb[2 * i + 1] = e4m3x2_to_bf16x2(wq[i] >> 16);
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m >= p.M) continue;
                const uint16_t* xm = xk + (long long)m * p.K + 16 * c;
                const uint4 x0 = ldg128(xm), x1 = ldg128(xm + 8);
                float a = part[m];
                a = fma2_bf16(wb[0], x0.x, a);
                a = fma2_bf16(wb[1], x0.y, a);
                a = fma2_bf16(wb[2], x0.z, a);
                a = fma2_bf16(wb[3], x0.w, a);
                a = fma2_bf16(wb[4], x1.x, a);
                a = fma2_bf16(wb[5], x1.y, a);
                a = fma2_bf16(wb[6], x1.z, a);
                a = fma2_bf16(wb[7], x1.w, a);
                part[m] = a;
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = fmaf(part[m], scale, acc[m]);
    }

    // Finish a run: thread (w < 4, l) stores weight row 32 w + l for every
    // token (SwiGLU on a finished tile: gate row l < 8 of each 16-row group
    // pairs with up row l + 8, lane l ^ 8; argmax: the warp's best per token
    // goes to its row sbest[16]).
    __device__ __forceinline__ void write_rows(const LinearParams& p, float* slot, int n0, int warp,
                                               int lane, unsigned long long* sbest) {
        if (warp >= 4) return;
        const int row = warp * 32 + lane;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float v = acc[m];
            if (p.act == 1 && !slot) {
                const float up = __shfl_xor_sync(0xffffffffu, v, 8);
                if ((lane & 8) == 0 && m < p.M && n0 + row < p.N) write_swiglu(p, m, n0 + row, v, up);
            } else if (p.act == 2 && !slot) {
                unsigned long long k = 0;
                if (m < p.M && n0 + row < p.N) k = argmax_key(write_output(p, m, n0 + row, v), n0 + row);
                k = warp_max_key(k, 1);
                if (lane == 0 && m < p.M) sbest[m] = max_u64(sbest[m], k);
            } else {
                put_value(p, slot, n0, m, row, v);
            }
        }
    }
};

template <int DT, int FAM, int MT>
struct ConsumerOf {
    using type = SimtConsumer<DT, MT>;
};
template <int DT, int MT>
struct ConsumerOf<DT, kTC, MT> {
    using type = TcConsumer<MT>;
};
template <int DT, int MT>
struct ConsumerOf<DT, kMMA, MT> {
    using type = MmaConsumer<DT, MT>;
};

// ------------------------------------------------------------------ FP8 activation copy

// The exact f16 copy of x for the FP8 path, one (K block kb, token slot tok)
// pair per warp: lane `lane` holds the bf16 values of columns 4 lane ..
// 4 lane + 3 of the block in v (zero for tok >= M).  The block is scaled by
// 2^(141 - e), e the largest biased exponent of its values, so that its
// largest magnitude lands in [2^14, 2^15); every value is then exact in f16
// if no non-zero value has a biased exponent below e - 31 (f16 subnormals keep
// 8 significant bits down to 2^-17) and none is an infinity or NaN.
// unscale[kb][tok] = 2^(e - 141) (1 for an all-zero block and for the token
// slots M <= tok < mtb), or 0 when the block is not exact in f16.  xh is
// [K block][half][mtb token rows][64], rows tok >= M zero; within every group
// of 16 columns the values sit in the order the FP8 MMA fragments take them
// (position 2t + j holds column 4t + j and position 2t + 8 + j holds column
// 4t + 2 + j, t < 4, j < 2), so that a plain ldmatrix of a token row yields
// the B fragment matching the e4m3 codes 4t .. 4t + 3 a thread holds for the
// A operand.  The whole warp calls it with the same (kb, tok).
__device__ __forceinline__ void write_x_copy_pair(uint16_t* __restrict__ xh, float* __restrict__ unscale,
                                                  int M, int mtb, int kb, int tok, int lane, uint2 v) {
    // This lane's 4 columns 4t .. 4t + 3 (t = lane % 4) of 16-column group
    // (lane % 16) / 4 of half lane / 16 go to positions 2t, 2t + 1 and
    // 2t + 8, 2t + 9 of that group.
    const long long row = (((long long)kb * 2 + (lane >> 4)) * mtb + tok) * 64 + ((lane & 15) >> 2) * 16;
    uint16_t* d0 = xh + row + 2 * (lane & 3);
    uint16_t* d1 = d0 + 8;
    if (tok >= M) {
        if (tok < mtb) {
            *reinterpret_cast<uint32_t*>(d0) = 0u;
            *reinterpret_cast<uint32_t*>(d1) = 0u;
        }
        if (lane == 0) unscale[kb * kUnscaleStride + tok] = 1.f;
        return;
    }
    const uint32_t b[4] = {v.x & 0xffffu, v.x >> 16, v.y & 0xffffu, v.y >> 16};
    unsigned emax = 0, emin = 255;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const unsigned mag = b[i] & 0x7fffu;
        const unsigned e = mag >> 7;
        emax = e > emax ? e : emax;
        const unsigned ez = mag ? e : 255u;      // exact zeros do not bound the range
        emin = ez < emin ? ez : emin;
        bad |= (e == 255u);
    }
    emax = warp_max_u32(emax);
    emin = warp_min_u32(emin);
    const bool ok = !__any_sync(0xffffffffu, bad) &&
                    (emax == 0u || (emax >= 15u && emin + 31u >= emax));
    const float f = (ok && emax) ? __uint_as_float((268u - emax) << 23) : 0.f;
    const float x0 = __uint_as_float(v.x << 16) * f, x1 = __uint_as_float(v.x & 0xffff0000u) * f;
    const float x2 = __uint_as_float(v.y << 16) * f, x3 = __uint_as_float(v.y & 0xffff0000u) * f;
    *reinterpret_cast<uint32_t*>(d0) = f32x2_to_f16x2(x0, x1);
    *reinterpret_cast<uint32_t*>(d1) = f32x2_to_f16x2(x2, x3);
    if (lane == 0)
        unscale[kb * kUnscaleStride + tok] =
            !ok ? 0.f : (emax ? __uint_as_float((emax - 14u) << 23) : 1.f);
}

// The tensor-memory family's copy of x: three e4m3 parts per value, so that
// the 5th-generation tensor cores multiply e4m3 weights by e4m3 activations
// (kind::f8f6f4) with every product exact.  Per (K block kb, token slot tok),
// with e the largest biased exponent of the block's bf16 values, x is scaled
// by f = 2^(134 - e) (its largest magnitude lands in [2^7, 2^8)) and split:
// p0 = e4m3(x f), p1 = e4m3((x f - p0) 2^4), p2 = e4m3(((x f - p0) 2^4 - p1) 2^4),
// each rounded to nearest even.  x f = p0 + p1 2^-4 + p2 2^-8 exactly when the
// last remainder is zero: every non-zero value within about 17 binades of
// the block's largest.  unscale[kb][tok] = 2^(e - 134) (1 for an all-zero
// block and for the token slots M <= tok < mtb), or 0 when the split is not
// exact (the block then takes the exact bf16 route).  Layout: rows of 128
// bytes, [K block][part][mtb token slots], rows tok >= M zero; byte k of a
// row is column k of the block, so a SWIZZLE_128B tensor copy of rows lands
// as the K-major B operand of the MMA.  Lane `lane` holds columns 4 lane ..
// 4 lane + 3 of the block in v; the whole warp calls it with the same (kb, tok).
__device__ __forceinline__ void f16x2_to_f32x2(uint32_t h2, float& lo, float& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
}

__device__ __forceinline__ void e4m3x4_to_f32x4(uint32_t four, float (&v)[4]) {
    uint32_t lo, hi;
    e4m3x4_to_f16x2x2(four, lo, hi);
    f16x2_to_f32x2(lo, v[0], v[1]);
    f16x2_to_f32x2(hi, v[2], v[3]);
}

__device__ __forceinline__ void write_x_parts_pair(uint8_t* __restrict__ xp, float* __restrict__ unscale,
                                                   int M, int mtb, int kb, int tok, int lane, uint2 v) {
    uint8_t* row0 = xp + ((long long)kb * 3 * mtb + tok) * 128 + 4 * lane;
    const long long part = (long long)mtb * 128;           // bytes between the parts' rows
    if (tok >= M) {
        if (tok < mtb) {
#pragma unroll
            for (int q = 0; q < 3; ++q) *reinterpret_cast<uint32_t*>(row0 + q * part) = 0u;
        }
        if (lane == 0) unscale[kb * kUnscaleStride + tok] = 1.f;
        return;
    }
    const uint32_t b[4] = {v.x & 0xffffu, v.x >> 16, v.y & 0xffffu, v.y >> 16};
    unsigned emax = 0;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const unsigned e = (b[i] & 0x7fffu) >> 7;
        emax = e > emax ? e : emax;
        bad |= (e == 255u);
    }
    emax = warp_max_u32(emax);
    bad = __any_sync(0xffffffffu, bad) || (emax != 0u && emax < 8u);
    // 2^(134 - e) as an fp32 bit pattern (0 for an all-zero or unusable block)
    const float f = (!bad && emax) ? __uint_as_float((261u - emax) << 23) : 0.f;
    float x[4], r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(b[i] << 16) * f;
    uint32_t q[3];
    bool rest = false;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        q[k] = f32x2_to_e4m3x2(x[0], x[1]) | (f32x2_to_e4m3x2(x[2], x[3]) << 16);
        e4m3x4_to_f32x4(q[k], r);
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = (x[i] - r[i]) * 16.f;      // exact
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) rest |= (x[i] != 0.f);
    const bool ok = !bad && !__any_sync(0xffffffffu, rest);
#pragma unroll
    for (int k = 0; k < 3; ++k) *reinterpret_cast<uint32_t*>(row0 + k * part) = q[k];
    if (lane == 0)
        unscale[kb * kUnscaleStride + tok] =
            !ok ? 0.f : (emax ? __uint_as_float((emax - 7u) << 23) : 1.f);
}

// ------------------------------------------------------------------ fix-up

// Last arriver of a split tile: y[m][n0 + rr] = the sum, in ascending segment
// order, of the partial rows the tile's segments j_first .. j_last stored
// (slot 1 of j_first when that segment began in an earlier tile, else slot 0;
// slot 0 of every later one), + bias.  The order is fixed, so the result does
// not depend on which CTA arrives last.  All loads are issued before the first
// add (float4 rows, up to kBatch segments in flight): one L2 round trip per
// kBatch segments instead of one per load.  Thread tid owns rows 4 (g % 32) ..
// + 3 of token g / 32 for g = tid (and tid + 256 when 16 tokens are staged),
// so a warp's lanes share one token (argmax: one warp reduction per token;
// the next layer's activation copy: one block per warp, p.xh_next).
// kLocal: the tile was covered whole by one segment of this CTA, whose warps
// stored its rows in the CTA's own slot `local` (no other CTA involved, plain
// cached loads after a CTA-scope barrier).
template <int MTB, bool kLocal = false>
__device__ __forceinline__ void fixup_tile(const LinearParams& p, int tile, int j_first, int j_last,
                                           int tid, unsigned long long* sbest,
                                           const float* local = nullptr) {
    constexpr int kBatch = 8;
    constexpr int kG = MTB > 8 ? 2 : 1;                       // row groups per thread
    constexpr long long kStride = 2LL * MTB * kBN;            // floats between segments' slot 0
    const int n0 = tile * kBN;
    const int sl_first = kLocal ? 0 : ((seg_begin(p, j_first) / p.UT == tile) ? 0 : 1);
    const int nseg = kLocal ? 1 : j_last - j_first + 1;
    const int ng = p.M * (kBN / 4);
    const float* first = kLocal ? local : p.partials + ((long long)j_first * 2 + sl_first) * MTB * kBN;
    int off[kG];
    bool has[kG];
    float4 v[kG];
#pragma unroll
    for (int i = 0; i < kG; ++i) {
        const int g = tid + i * kConsumerThreads;
        has[i] = g < ng;
        off[i] = (g >> 5) * kBN + (g & 31) * 4;
        v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int j0 = 0; j0 < nseg; j0 += kBatch) {
        float4 a[kG][kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int j = j0 + q;
            const float* src = j == 0 ? first : p.partials + (long long)(j_first + j) * kStride;
#pragma unroll
            for (int i = 0; i < kG; ++i) {
                if (kLocal)
                    a[i][q] = (has[i] && j < nseg) ? *reinterpret_cast<const float4*>(src + off[i])
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                else
                    a[i][q] = (has[i] && j < nseg) ? ld_cg_f32x4(src + off[i]) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            if (j0 + q >= nseg) break;
#pragma unroll
            for (int i = 0; i < kG; ++i) {
                if (j0 + q == 0) {
                    v[i] = a[i][q];
                } else {
                    v[i].x += a[i][q].x;
                    v[i].y += a[i][q].y;
                    v[i].z += a[i][q].z;
                    v[i].w += a[i][q].w;
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kG; ++i) {
        const int g = tid + i * kConsumerThreads;
        if (g >= kG * kConsumerThreads) break;
        const int m = g >> 5, rr = (g & 31) * 4;
        const float vv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        unsigned long long k = 0;
        uint32_t yb[4] = {0u, 0u, 0u, 0u};                   // the bf16 outputs
        if (has[i]) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (n0 + rr + c < p.N) {
                    const float vb = write_output(p, m, n0 + rr + c, vv[c]);
                    yb[c] = f32_to_bf16_rne(vb);
                    if (p.act == 2) k = max_u64(k, argmax_key(vb, n0 + rr + c));
                }
            }
        }
        // The next layer's exact f16 copy of this block (K block `tile` of its
        // x, token m): N % 128 == 0 there, so all 128 columns are outputs.
        if (p.xh_next)
            write_x_copy_pair(p.xh_next, p.us_next, p.M, MTB, tile, m, tid & 31,
                              make_uint2(yb[0] | (yb[1] << 16), yb[2] | (yb[3] << 16)));
        if (p.act == 2 && m < p.M) {                         // the warp's 32 lanes share m
            k = warp_max_key(k, 1);
            if ((tid & 31) == 0) sbest[m] = max_u64(sbest[m], k);
        }
    }
}

// The same for a SwiGLU tile.  Thread tid < 16 M owns, for token tid / 16, the
// gate rows 16 b + 4 h .. + 3 and their up rows (+ 8), b = (tid / 2) % 8,
// h = tid % 2: four outputs, both sums in ascending segment order.
template <int MTB>
__device__ __forceinline__ void fixup_tile_swiglu(const LinearParams& p, int tile, int j_first,
                                                  int j_last, int tid) {
    constexpr int kBatch = 8;
    constexpr long long kStride = 2LL * MTB * kBN;
    if (tid >= p.M * 16) return;
    const int n0 = tile * kBN;
    const int sl_first = (seg_begin(p, j_first) / p.UT == tile) ? 0 : 1;
    const int nseg = j_last - j_first + 1;
    const int m = tid >> 4, rr = ((tid >> 1) & 7) * 16 + (tid & 1) * 4;
    const int off = m * kBN + rr;
    const float* first = p.partials + ((long long)j_first * 2 + sl_first) * MTB * kBN;
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
    for (int j0 = 0; j0 < nseg; j0 += kBatch) {
        float4 ag[kBatch], au[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int j = j0 + q;
            const float* src = j == 0 ? first : p.partials + (long long)(j_first + j) * kStride;
            const bool in = j < nseg;
            ag[q] = in ? ld_cg_f32x4(src + off) : make_float4(0.f, 0.f, 0.f, 0.f);
            au[q] = in ? ld_cg_f32x4(src + off + 8) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            if (j0 + q >= nseg) break;
            if (j0 + q == 0) {
                g = ag[q];
                u = au[q];
            } else {
                g.x += ag[q].x; g.y += ag[q].y; g.z += ag[q].z; g.w += ag[q].w;
                u.x += au[q].x; u.y += au[q].y; u.z += au[q].z; u.w += au[q].w;
            }
        }
    }
    if (n0 + rr >= p.N) return;                        // N % 16 == 0: the group is whole
    write_swiglu(p, m, n0 + rr, g.x, u.x);
    write_swiglu(p, m, n0 + rr + 1, g.y, u.y);
    write_swiglu(p, m, n0 + rr + 2, g.z, u.z);
    write_swiglu(p, m, n0 + rr + 3, g.w, u.w);
}

// ------------------------------------------------------------------ kernel

template <int DT, int FAM, int MT>
__global__ void __launch_bounds__(threads_for(DT, FAM), min_blocks_for(DT, FAM, MT))
linear_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_s, const LinearParams p) {
    using Consumer = typename ConsumerOf<DT, FAM, MT>::type;
    constexpr int MTB = XRows<MT>::v;
    constexpr int W_UNIT = TileBytes<DT>::w;                 // weights of one unit
    // activations of one unit: bf16 x, the f16 copy, or (tensor-memory
    // family) the three e4m3 parts of every token slot, 128 bytes per row
    constexpr int X_UNIT = FAM == kTC ? TcShape<MTB>::rows * 128 : MTB * kBK * 2;
    constexpr int X_STAGE = DT == kBF16 ? X_UNIT : kMaxUnitsPerStage * X_UNIT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const SmemLayout L = smem_layout(DT, FAM, MT, S);
    uint8_t* sW = smem + L.w;
    uint8_t* sX = smem + L.x;
    StageHeader* hdr = reinterpret_cast<StageHeader*>(smem + L.hdr);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + S;
    uint64_t* written = empty + S;    // [2] consumer warps -> ticket warp (count 8)
    uint64_t* result = written + 2;   // [2] ticket warp -> consumer warps (count 1)
    uint64_t* xch = result + 2;       // consumer warps -> each other (count 8): a whole
                                      //   tile's rows are in the CTA's slot
    uint64_t* mma_done = xch + 1;     // [2] tensor-memory family: a stage's MMAs completed
    uint64_t* tmem_free = mma_done + 2;   // [2] warps 0-3 have read a TMEM buffer (count 4)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tmem_free + 2);
    volatile RunSlot* runs = reinterpret_cast<volatile RunSlot*>(smem + L.runs);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.runs + 2 * sizeof(RunSlot));
    // argmax (act = 2): each consumer warp's best key per token
    unsigned long long* sbest = reinterpret_cast<unsigned long long*>(smem + L.best) + (threadIdx.x >> 5) * 16;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int KB = p.KB;
    const int UT = p.UT;
    constexpr int kUnitKB = DT == kBF16 ? 1 : kMaxUnitsPerStage;   // K blocks per unit
    const WaitCtl err{p.err, p.wait_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            // tensor-memory family: the stage's MMAs (one commit) read it too
            mbar_init(smem_u32(&empty[s]), kConsumerWarps + (FAM == kTC ? 1 : 0));
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&written[b]), kConsumerWarps);
            mbar_init(smem_u32(&result[b]), 1);
        }
        mbar_init(smem_u32(xch), kConsumerWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&mma_done[b]), 1);
            mbar_init(smem_u32(&tmem_free[b]), 4);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
        griddep_launch_dependents();
    }
    if (warp == kLoaderWarp && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
        if constexpr (DT == kFP8) prefetch_tmap(&tm_s);
    }
    if constexpr (FAM == kTC) {
        // The accumulators of two stages (two units each) in tensor memory.
        // One CTA per SM, so the columns are free; this warp frees them
        // before the CTA exits, on every path.
        if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), TcShape<MTB>::cols);
        tc_fence_before_sync();
    }
    __syncthreads();
    if constexpr (FAM == kTC) tc_fence_after_sync();
    // Everyone but the loader sleeps until the previous kernel on the stream
    // has finished (a hardware wait, no polling while it runs).
    if (warp != kLoaderWarp) griddep_wait();

    // ---------------------------------------------------------------- MMA warp
    // Tensor-memory family: for each stage, in order, one thread issues the
    // UMMAs of its units (4 K steps of 32 per unit, M = 128 weight rows, N =
    // the activation parts) into TMEM buffer (stage number & 1), then commits
    // twice: to mma_done of that buffer (warps 0-3 read the results) and to
    // the stage's empty barrier (its buffer may be refilled once the MMAs have
    // read it).  A buffer is reused only after warps 0-3 freed it.
    if constexpr (FAM == kTC) {
        if (warp == kMmaWarp) {
            constexpr int NU = TcShape<MTB>::n;
            constexpr uint32_t idesc = umma_idesc_e4m3(NU);
            const uint32_t tmem = *tmem_slot;
            if (lane == 0) {
                long long seq = 0;
                int s = 0;
                uint32_t ph = 0;
                while (true) {
                    if (!mbar_wait_bounded(smem_u32(&full[s]), ph, err, kErrConsumerWait)) {
                        *abort_flag = 1;
                        break;
                    }
                    if ((hdr[s].flags & kDone) || *abort_flag) break;
                    const int nkb = hdr[s].nkb;
                    const int b = (int)(seq & 1);
                    if (seq >= 2 && !mbar_wait_bounded(smem_u32(&tmem_free[b]), (uint32_t)(((seq >> 1) - 1) & 1),
                                                       err, kErrRunWait)) {
                        *abort_flag = 1;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sw = smem_u32(sW + (size_t)s * kStageWBytes);
                    const uint32_t sx = smem_u32(sX + (size_t)s * X_STAGE);
                    for (int u = 0; u < nkb; ++u) {
                        const uint32_t d = tmem + (uint32_t)((b * 2 + u) * NU);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            umma_e4m3(d, umma_desc_sw128(sw + u * W_UNIT + 32 * j),
                                      umma_desc_sw128(sx + u * X_UNIT + 32 * j), idesc, j > 0);
                    }
                    umma_commit(smem_u32(&mma_done[b]));
                    umma_commit(smem_u32(&empty[s]));
                    ++seq;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                // Free the columns only once the last MMAs have completed and
                // warps 0-3 have read their results (bounded waits).
                if (seq >= 1)
                    mbar_wait_bounded(smem_u32(&mma_done[(seq - 1) & 1]), (uint32_t)(((seq - 1) >> 1) & 1), err,
                                      kErrDrainWait);
                for (long long q = seq >= 2 ? seq - 2 : 0; q < seq; ++q)
                    mbar_wait_bounded(smem_u32(&tmem_free[q & 1]), (uint32_t)((q >> 1) & 1), err, kErrDrainWait);
            }
            __syncwarp();
            tc_fence_after_sync();
            tmem_dealloc(tmem, TcShape<MTB>::cols);
            return;
        }
    }

    // ---------------------------------------------------------------- ticket warp
    // For each split run, in order: wait until all consumer warps have stored
    // their partial rows, take the tile's ticket (acquire-release at GPU scope:
    // publishes those rows, and for the last arriver makes every other
    // contributor's rows visible), publish the outcome.
    if (warp == kTicketWarp) {
        if (lane == 0) {
            uint32_t wph = 0u;        // phase parity of written[b] in bit b
            for (int r = 0;; ++r) {
                const int b = r & 1;
                if (!mbar_wait_bounded(smem_u32(&written[b]), (wph >> b) & 1u, err, kErrRunWait))
                    break;
                wph ^= 1u << b;
                const int tile = runs[b].tile;
                if (tile < 0) break;
                const int old = atom_add_acq_rel_gpu(&p.tickets[tile], 1);
                runs[b].last = (old == runs[b].jl - runs[b].jf) ? tile : -1;
                mbar_arrive(smem_u32(&result[b]));
            }
        }
        return;
    }

    // ---------------------------------------------------------------- loader
    if (warp == kLoaderWarp) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            long long issued = 0;     // stages issued
            bool ok = true;
            // K blocks of unit ku of a tile: kb = ku * kUnitKB, and one or two.
            auto blocks_of = [&](int ku) -> int {
                if constexpr (DT == kFP8) return ku * 2 + 1 < KB ? 2 : 1;
                else return 1;
            };
            auto issue_w = [&](int s, int tile, int kb, int nkb) {
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t dw = smem_u32(sW + (size_t)s * kStageWBytes);
                if constexpr (DT == kBF16) {
                    tma_load_2d(dw, &tm_w, bar, kb * kBK, tile * kBN, pol_w);
                    tma_load_2d(dw + kBN * 128, &tm_w, bar, kb * kBK + 64, tile * kBN, pol_w);
                } else {
                    for (int u = 0; u < nkb; ++u)
                        tma_load_2d(dw + u * W_UNIT, &tm_w, bar, (kb + u) * kBK, tile * kBN, pol_w);
                    // The block scales of K blocks kb, kb + 1 (elements e, e + 1
                    // of the scales map): one box of 8 from e rounded down to a
                    // multiple of 4 (16 bytes) holds both.
                    const int e = p.scale_off + tile * KB + kb;
                    tma_load_1d(smem_u32(&hdr[s].scale8[0]), &tm_s, bar, e & ~3);
                }
            };
            // Activations of the stage.  bf16: x itself (two 64-column boxes).
            // FP8: the prep kernel's f16 copy, laid out [K block][half][MTB][64],
            // so one box of 4 MTB rows holds K blocks kb and kb + 1 (rows past
            // the end read as zero), and the unscale factors by one bulk copy.
            // Both are written by the prep kernel: only after the wait.
            auto issue_x = [&](int s, int kb, int nkb) {
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t dx = smem_u32(sX + (size_t)s * X_STAGE);
                if constexpr (DT == kFP8) {
                    bulk_load(smem_u32(&hdr[s].unscale[0][0]), p.unscale + (long long)kb * kUnscaleStride,
                              (uint32_t)(nkb * kUnscaleStride * 4), bar);
                    if constexpr (FAM == kTC)     // the parts of K blocks kb, kb + 1: 2 x 3 MTB rows
                        tma_load_2d(dx, &tm_x, bar, 0, kb * TcShape<MTB>::rows, pol_x);
                    else
                        tma_load_2d(dx, &tm_x, bar, 0, kb * 2 * MTB, pol_x);
                } else {
                    tma_load_2d(dx, &tm_x, bar, kb * kBK, 0, pol_x);
                    tma_load_2d(dx + MTB * 128, &tm_x, bar, kb * kBK + 64, 0, pol_x);
                }
            };
            // Header + block scales + arrival for unit (tile, ku): K blocks kb ..
            // kb + nkb - 1; `left` = units left in the segment including this one.
            // No division on this path.  The expected bytes include the copies
            // issued later (x, unscale), so the stage cannot complete before they
            // land.
            auto open_stage = [&](int s, int tile, int ku, int seg, bool seg_first, long long left) {
                const int kb = ku * kUnitKB, nkb = blocks_of(ku);
                int fl = 0;
                if (seg_first || ku == 0) fl |= kRunFirst;
                if (left == 1 || ku == UT - 1) fl |= kRunLast;
                sts128(smem_u32(&hdr[s].tile), tile, kb, seg, fl);
                hdr[s].nkb = nkb;
                const uint32_t bar = smem_u32(&full[s]);
                uint32_t bytes = 0;
                if constexpr (DT == kFP8) {
                    hdr[s].soff = (p.scale_off + tile * KB + kb) & 3;   // see issue_w
                    bytes = nkb * (W_UNIT + kUnscaleStride * 4) + X_STAGE + 8 * 4;
                } else {
                    bytes = W_UNIT + X_UNIT;
                }
                mbar_arrive_expect_tx(bar, bytes);
            };

            // Test hook for the bounded waits: CTA 0 opens its p.withhold-th
            // stage (the barrier expects the bytes) but never issues the
            // copies that would fill it, so every wait on that stage runs out
            // with nothing in flight for it.
            auto withheld = [&](long long idx) -> bool {
                return p.withhold > 0 && blockIdx.x == 0 && idx + 1 == p.withhold;
            };
            int seg = blockIdx.x;
            long long u0 = seg_begin(p, seg);
            long long u1 = seg_begin(p, seg + 1);
            int tile = (int)(u0 / UT), ku = (int)(u0 % UT);
            long long left = u1 - u0;
            // Weights and scales are never written by the previous kernel when
            // early_stages is set: fill that many stages' weight tiles before
            // waiting for it (more delays the first activation copy when the
            // previous kernel is short); everything else waits.
            int pre = 0;
            if (p.early_stages > 0) {
                int ptile = tile, pku = ku;
                for (; pre < S && pre < p.early_stages && pre < left; ++pre) {
                    open_stage(pre, ptile, pku, seg, pre == 0, left - pre);
                    if (!withheld(pre)) issue_w(pre, ptile, pku * kUnitKB, blocks_of(pku));
                    if (++pku == UT) { pku = 0; ++ptile; }
                }
            }
            griddep_wait();
            for (int st = 0; st < pre; ++st) {
                if (!withheld(st)) issue_x(st, ku * kUnitKB, blocks_of(ku));
                if (++ku == UT) { ku = 0; ++tile; }
            }
            left -= pre;
            issued = pre;
            // Stage and ring pass of stage `issued`, kept incrementally (the stage
            // count is a run-time value: no division on this path).
            int ls = pre;
            uint32_t lph = 0;
            if (ls == S) { ls = 0; lph = 1; }
            bool seg_first = pre == 0;
            while (ok) {
                for (; left > 0; --left) {
                    if (issued >= S &&
                        !mbar_wait_bounded(smem_u32(&empty[ls]), lph ^ 1u, err, kErrProducerWait)) {
                        ok = false;
                        *abort_flag = 1;
                        break;
                    }
                    open_stage(ls, tile, ku, seg, seg_first, left);
                    if (!withheld(issued)) {
                        issue_w(ls, tile, ku * kUnitKB, blocks_of(ku));
                        issue_x(ls, ku * kUnitKB, blocks_of(ku));
                    }
                    seg_first = false;
                    if (++ku == UT) { ku = 0; ++tile; }
                    ++issued;
                    if (++ls == S) { ls = 0; lph ^= 1u; }
                }
                if (!ok) break;
                if (p.n_segments == G) break;      // static partition: nothing to claim
                // Claim only when at most kClaimDepth issued stages are still
                // unconsumed, so that no CTA holds a long backlog when the
                // shared segments run out: wait for stage issued - kClaimDepth
                // to be released (its ring slot and pass follow from ls, lph).
                if (issued >= kClaimDepth && kClaimDepth < S) {
                    const bool wrap = ls < kClaimDepth;
                    const int qs = wrap ? ls - kClaimDepth + S : ls - kClaimDepth;
                    if (!mbar_wait_bounded(smem_u32(&empty[qs]), wrap ? lph ^ 1u : lph, err,
                                           kErrProducerWait)) {
                        *abort_flag = 1;
                        break;
                    }
                }
                // Claim the next segment after the first wave; the unsigned range
                // check keeps every index in bounds even with a corrupted counter.
                const unsigned claimed = (unsigned)atomicAdd(&p.counter[0], 1);
                if (claimed >= (unsigned)(p.n_segments - G)) break;
                seg = G + (int)claimed;
                u0 = seg_begin(p, seg);
                u1 = seg_begin(p, seg + 1);
                tile = (int)(u0 / UT);
                ku = (int)(u0 % UT);
                left = u1 - u0;
                seg_first = true;
            }
            // Tell the consumers there is no more work.
            {
                if (issued < S ||
                    mbar_wait_bounded(smem_u32(&empty[ls]), lph ^ 1u, err, kErrProducerWait)) {
                    hdr[ls].flags = kDone;
                    mbar_arrive(smem_u32(&full[ls]));
                    ++issued;
                } else {
                    *abort_flag = 1;
                }
            }
            // The last CTA to finish claiming re-arms the counter for the next call
            // (the fence orders this CTA's last claim before its count).
            __threadfence();
            if (atomicAdd(&p.counter[1], 1) == G - 1) {
                __threadfence();
                p.counter[0] = 0;
                p.counter[1] = 0;
            }
            // Do not leave while copies into this CTA's shared memory may be in
            // flight: wait (bounded) for the last phase issued on every stage.
            for (int s = 0; s < S && s < issued; ++s) {
                const long long last = s + ((issued - 1 - s) / S) * S;
                mbar_wait_bounded(smem_u32(&full[s]), (uint32_t)((last / S) & 1), err,
                                  kErrDrainWait);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    Consumer c;
    c.reset();
    if (lane < 16) sbest[lane] = 0ull;
    __syncwarp();
    int run_kb0 = 0;
    int n_split = 0;                  // split runs handed to the ticket warp so far
    uint32_t rph = 0u;                // phase parity of result[b] in bit b
    int n_local = 0;                  // whole tiles finished through the CTA's slots (xh_next)
    long long tc_seq = 0;             // tensor-memory family: stages consumed (TMEM buffer, parities)
    const uint32_t tmem = FAM == kTC ? *tmem_slot : 0u;

    // Hand split run `tile` (partial rows already stored) to the ticket warp;
    // tile < 0 tells it that there are no more.
    auto hand_over = [&](int tile, int jf, int jl) {
        const int b = n_split & 1;
        if (threadIdx.x == 0) {
            runs[b].tile = tile;
            runs[b].jf = jf;
            runs[b].jl = jl;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&written[b]));
    };
    // Outcome of split run q: if it completed its tile, every consumer thread
    // helps finish the tile.  False if the wait gave up.
    auto settle = [&](int q) -> bool {
        const int b = q & 1;
        if (!mbar_wait_bounded(smem_u32(&result[b]), (rph >> b) & 1u, err, kErrRunWait))
            return false;
        rph ^= 1u << b;
        const int ft = runs[b].last;
        if (ft >= 0) {
            const long long tu0 = (long long)ft * UT;
            if (p.act == 1)
                fixup_tile_swiglu<MTB>(p, ft, seg_of(p, tu0), seg_of(p, tu0 + UT - 1), threadIdx.x);
            else
                fixup_tile<MTB>(p, ft, seg_of(p, tu0), seg_of(p, tu0 + UT - 1), threadIdx.x, sbest);
            if (threadIdx.x == 0) p.tickets[ft] = 0;
        }
        return true;
    };

    // Stage s and ring-pass parity ph of the stage being consumed, kept
    // incrementally (no division by the run-time stage count).
    int s = 0;
    uint32_t ph = 0;
    while (true) {
        if (!mbar_wait_bounded(smem_u32(&full[s]), ph, err, kErrConsumerWait)) {
            *abort_flag = 1;
            break;
        }
        const StageHeader& hd = hdr[s];
        const uint4 h4 = lds128(smem_u32(&hd.tile));      // tile, kb, seg, flags
        const int tile = (int)h4.x, kb = (int)h4.y, seg = (int)h4.z, flags = (int)h4.w;
        if ((flags & kDone) || *abort_flag) break;
        if (flags & kRunFirst) run_kb0 = kb;
        const uint32_t sw = smem_u32(sW + (size_t)s * kStageWBytes);
        const uint32_t sx = smem_u32(sX + (size_t)s * X_STAGE);
        int nkb = 1;
        if constexpr (FAM == kTC) {
            // Warps 0-3: a unit whose activation parts are not exact (an
            // unscale factor 0) is computed here from the weight tile, before
            // the buffer is released; the others are read from TMEM after
            // the MMA warp's commit, then the TMEM buffer is released.
            constexpr int NU = TcShape<MTB>::n;
            nkb = hd.nkb;
            float sc[2], u[2][MT];
            bool fb[2] = {false, false};
            if (warp < 4) {
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                    sc[uu] = hd.scale8[hd.soff + uu];
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        u[uu][m] = hd.unscale[uu][m];
                        if (uu < nkb && m < p.M) fb[uu] |= (u[uu][m] == 0.f);
                    }
                }
                const int row = warp * 32 + lane;
                if (fb[0]) c.add_exact_unit(sw, p, kb, row, sc[0]);
                if (nkb == 2 && fb[1]) c.add_exact_unit(sw + W_UNIT, p, kb + 1, row, sc[1]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (warp < 4) {
                const int b = (int)(tc_seq & 1);
                if (!mbar_wait_bounded(smem_u32(&mma_done[b]), (uint32_t)((tc_seq >> 1) & 1), err,
                                       kErrConsumerWait)) {
                    *abort_flag = 1;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t t0 = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * 2 * NU);
                if (!fb[0]) c.add_tmem_unit(t0, u[0], sc[0]);
                if (nkb == 2 && !fb[1]) c.add_tmem_unit(t0 + NU, u[1], sc[1]);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&tmem_free[b]));
            }
            ++tc_seq;
        } else {
            if constexpr (DT == kFP8) {
                nkb = hd.nkb;
                const int so = hd.soff;
                c.consume(sw, sx, hd.scale8[so], hd.unscale[0], kb, p, warp, lane);
                if (nkb == 2)
                    c.consume(sw + W_UNIT, sx + X_UNIT, hd.scale8[so + 1], hd.unscale[1], kb + 1, p, warp, lane);
            } else {
                c.consume(sw, sx, 1.f, nullptr, kb, p, warp, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        }

        if (flags & kRunLast) {
            // This run of `tile` is complete: store its rows (y, or the slot).
            const bool whole = (run_kb0 == 0) && (kb + nkb == KB);
            if (whole && p.xh_next) {
                // The next layer's activation copy is made from whole blocks
                // (one warp per token): the warps put the tile's rows in one of
                // the CTA's two slots, meet, and finish it like a split tile of
                // one segment.  The slots alternate; a warp reaches the meeting
                // of a tile only after finishing the tile before, so a slot is
                // never overwritten while it is read.
                float* slot = p.wslot + ((long long)blockIdx.x * 2 + (n_local & 1)) * MTB * kBN;
                c.write_rows(p, slot, tile * kBN, warp, lane, sbest);
                c.reset();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(xch));
                if (!mbar_wait_bounded(smem_u32(xch), (uint32_t)(n_local & 1), err, kErrRunWait)) {
                    *abort_flag = 1;
                    break;
                }
                fixup_tile<MTB, true>(p, tile, 0, 0, threadIdx.x, sbest, slot);
                ++n_local;
                if (++s == S) { s = 0; ph ^= 1u; }
                continue;
            }
            float* slot = nullptr;
            if (!whole) {
                const long long first_tile = seg_begin(p, seg) / UT;
                slot = p.partials + ((long long)seg * 2 + (tile == first_tile ? 0 : 1)) * MTB * kBN;
            }
            c.write_rows(p, slot, tile * kBN, warp, lane, sbest);
            c.reset();
            if (!whole) {
                // Hand this run over, then settle the previous split run (its
                // ticket has had a whole run to come back).
                int jf = 0, jl = 0;
                if (threadIdx.x == 0) {
                    const long long tu0 = (long long)tile * UT;
                    jf = seg_of(p, tu0);
                    jl = seg_of(p, tu0 + UT - 1);
                }
                hand_over(tile, jf, jl);
                ++n_split;
                if (n_split >= 2 && !settle(n_split - 2)) { *abort_flag = 1; break; }
            }
        }
        if (++s == S) { s = 0; ph ^= 1u; }
    }
    // Release the ticket warp and settle the last split run before leaving.
    if (!*abort_flag) {
        hand_over(-1, 0, 0);
        if (n_split >= 1) settle(n_split - 1);
    }
    // Argmax: every consumer warp merges its per-token best into the call's keys
    // (an atomic max: order-free); the last warp of the grid to do so turns them
    // into indices and values and leaves the keys and its counter at zero.
    if (p.act == 2 && !*abort_flag) {
        __syncwarp();
        if (lane < p.M) atomicMax(&p.best[lane], sbest[lane]);
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(&p.counter[2], 1) == (int)gridDim.x * kConsumerWarps - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            if (lane < p.M) {
                const unsigned long long k = atomicExch(&p.best[lane], 0ull);
                p.idx[lane] = (int)(0xffffffffu - (unsigned)(k & 0xffffffffu));
                if (p.maxval) p.maxval[lane] = argmax_key_value(k);
            }
            if (lane == 0) p.counter[2] = 0;
        }
    }
}

}  // namespace dl
