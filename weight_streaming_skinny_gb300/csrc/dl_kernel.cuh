// The decode-linear kernel: y[M,N] = x[M,K] . w[N,K]^T (+ bias), M <= 16.
//
// Work decomposition.  The weight matrix is cut into tiles of kBN = 128 rows;
// each tile's K range is cut into units of kBK = 128 columns (one FP8 scale
// block).  The U = tiles x k-blocks units, in tile-major order, are cut into
// contiguous segments by a partition fixed by (M, N, K, SM count) alone: a
// first wave of one large segment per CTA (about 5/8 of the work), then waves
// of segments that halve in size down to a small minimum.  A persistent grid
// of about one CTA per SM takes segment blockIdx.x of the first wave and then
// claims further segments, in order, from an atomic counter, so SMs that
// happen to stream faster take more of the small segments and all of them
// finish together.  This is the "split the long dimension across blocks so
// the whole chip streams weights" of "9% faster GLM-5.3-Flash prefill with
// GPU-to-GPU IPC" (section "TileLang: twice as fast, and no faster", where a
// 1..6-token step otherwise launches 16-96 blocks for 188 SMs), balanced at
// run time.
//
// Pipeline.  Warp 8 (one elected thread) streams units HBM -> shared memory
// with TMA tensor copies into a ring of `stages` buffers guarded by full/empty
// mbarriers; each buffer carries a header naming its unit (and, for FP8, the
// unit's block scale, copied asynchronously on the same barrier).  The weight
// tile is copied as 128 rows x 128 bytes with the 128-byte swizzle.  Warps 0-7
// each own 16 weight rows of the tile (the TileLang loop's T.Pipelined(...,
// num_stages=2), deepened to cover GB300's HBM latency).  Every weight byte is
// read from HBM exactly once per call.
//
// Consumer families:
//   SIMT: one weight row per lane (two lanes per row, one per K half), CUDA-core
//         fused multiply-adds with bf16 x bf16 -> fp32 products (the row-tiled
//         GEMV of "Developing a custom Qwen2.5 72B inference engine from
//         scratch", §6.1); a shuffle joins the two halves at the end of a run.
//   MMA:  warp-level mma.sync m16n8k16 -> fp32 with the weights as the 16-row A
//         operand and the (<= 16) tokens as the B operand (the
//         "T.gemm(A_s, B_h, acc, transpose_B=True)" of the TileLang loop).
//         bf16 weights feed a bf16 MMA directly.  FP8 weights are decoded by
//         the hardware e4m3 -> f16 convert (exact) and multiplied, in an f16
//         MMA, with a copy of x scaled by a power of two per (token, unit) so
//         that it is exact in f16; the power of two is removed from the fp32
//         partial.  Consumer warp w makes that copy for token w of the next
//         stage while the current one is consumed.  Units whose x cannot be
//         represented that way run the same products in a bf16 MMA instead.
// Two accumulator sets alternate over the K steps (shorter dependency chains);
// they are added in a fixed order.  The fp32 block scale multiplies each
// 128-wide K block's fp32 partial.
//
// Split-K fix-up.  Within one segment the units of one tile form a "run".  A
// run that covers its whole tile is finished on the spot: every warp rounds
// its own rows (+ bias) to bf16 and stores them.  Otherwise the warps store
// their fp32 partial rows in the workspace slot of the run's (segment,
// first-or-last tile) pair; after a CTA barrier one thread takes the tile's
// arrival ticket with an acquire-release atomic, whose result is looked at
// only at the next run end (or exit), so its latency overlaps the next units.
// The last run to arrive then has all warps sum the tile's slots in segment
// order (= ascending K), add the bias, round once and zero the slots and the
// ticket.  No CTA ever waits for another, and the order of every sum is fixed
// by the partition alone, so results are bitwise reproducible whichever CTA
// computed which segment.  Inside one GPU this plays the role of the
// row-parallel "partial sums, then all-reduce" of "Multi-GPU Inference and
// Serving at Scale", Example 3.
//
// Dependent launch.  The kernel lets the next kernel on the stream launch as
// soon as it starts (griddepcontrol.launch_dependents); all its threads but
// the loader sleep in griddepcontrol.wait until the previous kernel has
// finished, and the loader touches nothing that kernel may have written before
// that wait -- except, when `early_weights` is set (a later layer of one
// dl_decode_stream call, whose predecessor is this same kernel and never
// writes weights or scales), the weight tiles and scales of its first stages,
// which it prefetches while the previous layer drains.
//
// Every wait is bounded (mbarrier waits give up after ~2 s, set a bit of the
// device error word and make the CTA leave in an orderly way).
#pragma once

#include "dl_device.cuh"

namespace dl {

constexpr int kBN = 128;                 // weight rows per tile
constexpr int kBK = 128;                 // K columns per unit (one FP8 scale block)
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kMaxWaves = 24;

enum DType { kBF16 = 0, kFP8 = 1 };
enum Family { kSIMT = 1, kMMA = 2 };

// Stage header flags.
constexpr int kRunFirst = 1;   // first unit of a run (a run = one tile inside one segment)
constexpr int kRunLast = 2;    // last unit of a run
constexpr int kDone = 4;       // no more work: consumers leave

struct LinearParams {
    const uint16_t* bias;     // bf16 [N] or null
    uint16_t* y;              // bf16 [M][N]
    float* y_f32;             // fp32 [M][N] or null
    const float* scales;      // fp32 [ceil(N/128)][KB] (FP8)
    int* counter;             // [0]: segments claimed after the first wave, [1]: CTAs done
    int* tickets;             // [n_tiles] arrival counters (zero between calls)
    float* partials;          // [n_segments][2][MTB][kBN] fp32 (zero between calls)
    int M, N, K;
    int KB;                   // k-blocks per tile = ceil(K / 128)
    int n_tiles;
    long long units;          // n_tiles * KB
    int n_segments;
    int n_waves;              // the partition: wave w holds segments
    int wave_seg0[kMaxWaves + 1];     //   [wave_seg0[w], wave_seg0[w+1]), each of
    long long wave_unit0[kMaxWaves];  //   wave_size[w] units from wave_unit0[w]
    int wave_size[kMaxWaves];         //   (the very last segment ends at U)
    int stages;
    int early_weights;        // prefetch the first weight tiles before griddepcontrol.wait
    unsigned* err;            // device error word (bounded waits OR their bit in)
};

struct StageHeader {
    int tile;                 // unit held by the stage: weight rows 128*tile..
    int kb;                   //   and K block kb
    int seg;                  // segment it belongs to
    int flags;                // kRunFirst | kRunLast | kDone
    float scale;              // FP8 block scale of the unit (copied asynchronously)
    int pad[3];
};

template <int DT>
struct TileBytes {
    static constexpr int w = kBN * kBK * (DT == kBF16 ? 2 : 1);
};

template <int MT>
struct XRows {
    static constexpr int v = MT < 8 ? 8 : MT;   // token rows staged (zero-filled past M)
};

// Shared-memory layout of one CTA (offsets from a 1024-aligned base).  The
// host sizes the launch with the same function.
struct SmemLayout {
    int w, x, xh, hdr, unscale, bad, bars, flags, total;
};

__host__ __device__ constexpr SmemLayout smem_layout(int dtype, int family, int mt, int stages) {
    const int mtb = mt < 8 ? 8 : mt;
    const int wbytes = kBN * kBK * (dtype == kBF16 ? 2 : 1);
    const int xbytes = mtb * kBK * 2;
    const bool half_x = (dtype == kFP8 && family == kMMA);
    SmemLayout L{};
    L.w = 0;
    L.x = L.w + stages * wbytes;
    L.xh = L.x + stages * xbytes;
    L.hdr = L.xh + (half_x ? stages * xbytes : 0);
    L.unscale = L.hdr + stages * 32;
    L.bad = L.unscale + (half_x ? stages * 16 * 4 : 0);
    L.bars = L.bad + (half_x ? stages * 16 : 0);
    L.flags = L.bars + (3 * stages + 1) * 8;
    L.total = L.flags + 16;
    return L;
}

// Threads of a CTA: 8 consumer warps and the loader warp.
__host__ __device__ constexpr int threads_for(int, int) { return kConsumerThreads + 32; }

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

__device__ __forceinline__ void write_output(const LinearParams& p, int m, int n, float v) {
    if (p.bias) v += bf16_bits_to_f32(p.bias[n]);
    const long long o = (long long)m * p.N + n;
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

    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, uint32_t, const float*, bool,
                                            int warp, int lane, float scale) {
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
            float part[2][MT];
            uint32_t guard = 0;
            fp8_unit<false>(sw, xbase, row, h, sw8, part, guard);
            // A NaN code anywhere in the warp's unit: redo it with the decode
            // that keeps NaN (never taken for clamped weights).
            if (__any_sync(0xffffffffu, nan_guard_tripped(guard)))
                fp8_unit<true>(sw, xbase, row, h, sw8, part, guard);
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[0][m] = fmaf(part[0][m] + part[1][m], scale, acc[0][m]);
        }
    }

    template <bool kExactNaN>
    __device__ __forceinline__ void fp8_unit(uint32_t sw, uint32_t xbase, int row, int h, int sw8,
                                             float (&part)[2][MT], uint32_t& guard) {
        const uint32_t wbase = sw + row * 128;
#pragma unroll
        for (int m = 0; m < MT; ++m) part[0][m] = part[1][m] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cc = 4 * h + j;                  // 16-code chunk of the row
            const uint4 w = lds128(wbase + ((cc ^ sw8) << 4));
            const uint32_t wq[4] = {w.x, w.y, w.z, w.w};
            uint32_t wb[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if constexpr (kExactNaN) {
                    wb[2 * i] = e4m3x2_to_bf16x2(wq[i] & 0xffffu);
                    wb[2 * i + 1] = e4m3x2_to_bf16x2(wq[i] >> 16);
                } else {
                    wb[2 * i] = e4m3x2_to_bf16x2_fast(wq[i] & 0xffffu, guard);
                    wb[2 * i + 1] = e4m3x2_to_bf16x2_fast(wq[i] >> 16, guard);
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                // codes 16cc..16cc+15 pair with bf16 chunks 2j, 2j+1 of x box h
                const uint4 x0 = lds128(xbase + m * 128 + (((2 * j) ^ (m & 7)) << 4));
                const uint4 x1 = lds128(xbase + m * 128 + (((2 * j + 1) ^ (m & 7)) << 4));
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

    // Finish a run: join the accumulators and the two K halves, store the rows.
    __device__ __forceinline__ void write_rows(const LinearParams& p, float* slot, int n0, int warp,
                                               int lane) {
        const int row = warp * 16 + (lane & 15);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float mine = acc[0][m] + acc[1][m];
            const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
            if (lane < 16) put_value(p, slot, n0, m, row, mine + other);
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

    // sx: bf16 x tile of the stage; sxh: the same tile scaled exactly into
    // f16 (FP8 only); xunscale[tok]: the power of two that undoes the
    // scaling; exact_bf16: x of this unit is not exact in f16.
    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, uint32_t sxh,
                                            const float* xunscale, bool exact_bf16, int warp,
                                            int lane, float scale) {
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
            float part[2][NT][4];
            const int t = lane & 3;
            if (!exact_bf16) {
                fp8_unit_f16(abase, aswz, mat, sxh, lane, part);
            } else {
                uint32_t guard = 0;
                fp8_unit_bf16<false>(abase, aswz, mat, sx, lane, part, guard);
                if (__any_sync(0xffffffffu, nan_guard_tripped(guard)))
                    fp8_unit_bf16<true>(abase, aswz, mat, sx, lane, part, guard);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // f16 path: part was computed against x * 2^k; undo the (exact)
                // power of two, then apply the block scale.
                const float u0 = exact_bf16 ? 1.f : xunscale[8 * nt + 2 * t];
                const float u1 = exact_bf16 ? 1.f : xunscale[8 * nt + 2 * t + 1];
                acc[0][nt][0] = fmaf((part[0][nt][0] + part[1][nt][0]) * u0, scale, acc[0][nt][0]);
                acc[0][nt][1] = fmaf((part[0][nt][1] + part[1][nt][1]) * u1, scale, acc[0][nt][1]);
                acc[0][nt][2] = fmaf((part[0][nt][2] + part[1][nt][2]) * u0, scale, acc[0][nt][2]);
                acc[0][nt][3] = fmaf((part[0][nt][3] + part[1][nt][3]) * u1, scale, acc[0][nt][3]);
            }
        }
    }

    // One FP8 unit (this warp's 16 rows x 128 codes) as an f16 MMA against the
    // scaled f16 copy of x.  Step s is the 16-code chunk s of each row.  Thread
    // (g, t) receives codes 4t..4t+3 of its rows' chunk; they stand for
    // fragment columns {2t, 2t+1} and {2t+8, 2t+9}, so its B fragment is
    // x[token][16s + 4t .. 16s + 4t + 3], 8 bytes of the swizzled x box.
    __device__ __forceinline__ void fp8_unit_f16(uint32_t abase, int aswz, int mat, uint32_t sxh,
                                                 int lane, float (&part)[2][NT][4]) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[k][nt][i] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; s += 2) {
            uint32_t q[4];
            ldmatrix_x4(abase + (((s + (mat >> 1)) ^ aswz) << 4), q[0], q[1], q[2], q[3]);
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int step = s + ss;
                uint32_t A0, A1, A2, A3;
                e4m3x4_to_f16x2x2(q[2 * ss], A0, A2);       // row g
                e4m3x4_to_f16x2x2(q[2 * ss + 1], A1, A3);   // row g + 8
                const uint32_t xbox = sxh + (step >> 2) * (MT * 128);
                const int xc = 2 * (step & 3) + (t >> 1);   // logical 16-byte chunk
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = g + 8 * nt;
                    const uint2 xb = lds64(xbox + tok * 128 + ((xc ^ (tok & 7)) << 4) + ((t & 1) << 3));
                    mma_f16_16816(part[ss][nt], A0, A1, A2, A3, xb.x, xb.y);
                }
            }
        }
    }

    // The same products in a bf16 MMA against x as given, for units whose x is
    // not exact in f16.  kExactNaN selects the decode that keeps NaN codes.
    template <bool kExactNaN>
    __device__ __forceinline__ void fp8_unit_bf16(uint32_t abase, int aswz, int mat, uint32_t sx,
                                                  int lane, float (&part)[2][NT][4], uint32_t& guard) {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[k][nt][i] = 0.f;
#pragma unroll 1
        for (int s = 0; s < 8; s += 2) {
            uint32_t q[4];
            ldmatrix_x4(abase + (((s + (mat >> 1)) ^ aswz) << 4), q[0], q[1], q[2], q[3]);
#pragma unroll
            for (int ss = 0; ss < 2; ++ss) {
                const int step = s + ss;
                const uint32_t rlo = q[2 * ss], rhi = q[2 * ss + 1];
                uint32_t A0, A1, A2, A3;
                if constexpr (kExactNaN) {
                    A0 = e4m3x2_to_bf16x2(rlo & 0xffffu);
                    A2 = e4m3x2_to_bf16x2(rlo >> 16);
                    A1 = e4m3x2_to_bf16x2(rhi & 0xffffu);
                    A3 = e4m3x2_to_bf16x2(rhi >> 16);
                } else {
                    A0 = e4m3x2_to_bf16x2_fast(rlo & 0xffffu, guard);
                    A2 = e4m3x2_to_bf16x2_fast(rlo >> 16, guard);
                    A1 = e4m3x2_to_bf16x2_fast(rhi & 0xffffu, guard);
                    A3 = e4m3x2_to_bf16x2_fast(rhi >> 16, guard);
                }
                const uint32_t xbox = sx + (step >> 2) * (MT * 128);
                const int xc = 2 * (step & 3) + (t >> 1);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = g + 8 * nt;
                    const uint2 xb = lds64(xbox + tok * 128 + ((xc ^ (tok & 7)) << 4) + ((t & 1) << 3));
                    mma_bf16_16816(part[ss][nt], A0, A1, A2, A3, xb.x, xb.y);
                }
            }
        }
    }

    // Finish a run: add the accumulator sets and store the warp's rows.
    __device__ __forceinline__ void write_rows(const LinearParams& p, float* slot, int n0, int warp,
                                               int lane) {
        const int g = lane >> 2, t = lane & 3;
        const int row = warp * 16 + g;
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

template <int DT, int FAM, int MT>
struct ConsumerOf {
    using type = SimtConsumer<DT, MT>;
};
template <int DT, int MT>
struct ConsumerOf<DT, kMMA, MT> {
    using type = MmaConsumer<DT, MT>;
};

// Rescale one token's 128 bf16 x values of a unit exactly into f16 (FP8 MMA
// path).  Warp-cooperative: lane l converts 4 values in place of the
// swizzled tile layout (box l/16, 8 bytes at element (l%16)*4).  With e the
// largest biased exponent of the token's values, x * 2^(141 - e) has its
// largest magnitude in [2^14, 2^15); every value then fits f16 exactly if no
// non-zero value has a biased exponent below e - 31 (f16 subnormals keep 8
// significant bits down to 2^-17) and none is an infinity or NaN.  Writes the
// f16 values to sxh, 2^(e - 141) to *unscale and returns false when the
// token is not exact in f16.
template <int MTB>
__device__ __forceinline__ bool scale_token_to_f16(uint32_t sx, uint32_t sxh, int tok, int lane,
                                                   float* unscale) {
    const uint32_t off = (lane >> 4) * (MTB * 128) + tok * 128 +
                         ((((lane & 15) >> 1) ^ (tok & 7)) << 4) + ((lane & 1) << 3);
    const uint2 v = lds64(sx + off);
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
    sts64(sxh + off, f32x2_to_f16x2(x0, x1), f32x2_to_f16x2(x2, x3));
    if (lane == 0) *unscale = emax ? __uint_as_float((emax - 14u) << 23) : 1.f;
    return ok;
}

// Bounded barrier among the 8 consumer warps (lane 0 of each warp arrives on
// an mbarrier of count 8; every lane waits for the phase).  False if the wait
// gave up.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, int lane,
                                           unsigned* err) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(bar));
    const bool ok = mbar_wait_bounded(smem_u32(bar), phase, err, kErrGroupWait);
    phase ^= 1u;
    return ok;
}

// ------------------------------------------------------------------ fix-up

// Last arriver of a split tile: y[m][n0 + rr] = sum of the tile's partial
// slots in segment order (+ bias, one rounding); every slot is zeroed after
// it is read.  Only the first contributing segment can have started in an
// earlier tile (its slot 1); every later one started in this tile (slot 0),
// so their slots lie at a fixed stride and 16 loads are kept in flight.
template <int MTB>
__device__ __forceinline__ void fixup_tile(const LinearParams& p, int tile, int j_first, int j_last,
                                           int tid) {
    constexpr int kBatch = 16;
    constexpr long long kStride = 2LL * MTB * kBN;            // floats between segments' slot 0
    const int n0 = tile * kBN;
    const int sl_first = (seg_begin(p, j_first) / p.KB == tile) ? 0 : 1;
    for (int idx = tid; idx < p.M * kBN; idx += kConsumerThreads) {
        const int m = idx / kBN, rr = idx % kBN;
        float* first = p.partials + ((long long)j_first * 2 + sl_first) * MTB * kBN + m * kBN + rr;
        float v = ld_cg_f32(first);
        st_cg_f32(first, 0.f);
        float* base = p.partials + (long long)m * kBN + rr;
        for (int j0 = j_first + 1; j0 <= j_last; j0 += kBatch) {
            float val[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
                val[q] = (j0 + q <= j_last) ? ld_cg_f32(base + (long long)(j0 + q) * kStride) : 0.f;
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
                if (j0 + q <= j_last) v += val[q];       // ascending segment order
            // Leave the workspace all-zero: a later call with another shape may
            // place its arrival tickets over these bytes.
#pragma unroll
            for (int q = 0; q < kBatch; ++q)
                if (j0 + q <= j_last) st_cg_f32(base + (long long)(j0 + q) * kStride, 0.f);
        }
        if (n0 + rr < p.N) write_output(p, m, n0 + rr, v);
    }
}

// ------------------------------------------------------------------ kernel

template <int DT, int FAM, int MT>
__global__ void __launch_bounds__(threads_for(DT, FAM), min_blocks_for(DT, FAM, MT))
linear_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const LinearParams p) {
    using Consumer = typename ConsumerOf<DT, FAM, MT>::type;
    constexpr int MTB = XRows<MT>::v;
    constexpr int W_BYTES = TileBytes<DT>::w;
    constexpr int X_BYTES = MTB * kBK * 2;
    constexpr bool kHalfX = (DT == kFP8 && FAM == kMMA);
    constexpr int kLoaderWarp = kConsumerWarps;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    const SmemLayout L = smem_layout(DT, FAM, MT, S);
    uint8_t* sW = smem + L.w;
    uint8_t* sX = smem + L.x;
    uint8_t* sXh = smem + L.xh;                                          // [S][X_BYTES]
    StageHeader* hdr = reinterpret_cast<StageHeader*>(smem + L.hdr);
    float* unscale = reinterpret_cast<float*>(smem + L.unscale);       // [S][16]
    uint8_t* bad = smem + L.bad;                                        // [S][16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + S;
    uint64_t* xready = empty + S;
    uint64_t* gbar = xready + S;
    // flag[0..1]: the tile to finish at a run end, double-buffered by the group
    // barrier's phase so that thread 0 never overwrites a value a slower warp
    // has yet to read; flag[2]: abort.
    volatile int* flag = reinterpret_cast<volatile int*>(smem + L.flags);
    volatile int* abort_flag = flag + 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const int KB = p.KB;
    unsigned* err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
            mbar_init(smem_u32(&xready[s]), kConsumerWarps);
        }
        mbar_init(smem_u32(gbar), kConsumerWarps);
        flag[0] = flag[1] = -1;
        *abort_flag = 0;
        fence_mbarrier_init();
        griddep_launch_dependents();
    }
    if (warp == kLoaderWarp && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
    }
    __syncthreads();
    // Everyone but the loader sleeps until the previous kernel on the stream
    // has finished (a hardware wait, no polling while it runs).
    if (warp != kLoaderWarp) griddep_wait();

    // ---------------------------------------------------------------- loader
    if (warp == kLoaderWarp) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            long long issued = 0;
            bool ok = true;
            auto issue_w = [&](int s, int tile, int kb) {
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t dw = smem_u32(sW + (size_t)s * W_BYTES);
                tma_load_2d(dw, &tm_w, bar, kb * kBK, tile * kBN, pol_w);
                if constexpr (DT == kBF16)
                    tma_load_2d(dw + kBN * 128, &tm_w, bar, kb * kBK + 64, tile * kBN, pol_w);
            };
            auto issue_x = [&](int s, int kb) {
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t dx = smem_u32(sX + (size_t)s * X_BYTES);
                tma_load_2d(dx, &tm_x, bar, kb * kBK, 0, pol_x);
                tma_load_2d(dx + MTB * 128, &tm_x, bar, kb * kBK + 64, 0, pol_x);
            };
            // Header + scale + arrival for unit (tile, kb); `left` = units left in
            // the segment including this one.  No division on this path.
            auto open_stage = [&](int s, int tile, int kb, int seg, bool seg_first, long long left) {
                int fl = 0;
                if (seg_first || kb == 0) fl |= kRunFirst;
                if (left == 1 || kb == KB - 1) fl |= kRunLast;
                hdr[s].tile = tile;
                hdr[s].kb = kb;
                hdr[s].seg = seg;
                hdr[s].flags = fl;
                const uint32_t bar = smem_u32(&full[s]);
                if constexpr (DT == kFP8)
                    cp_async_4_mbar(smem_u32(&hdr[s].scale), p.scales + (long long)tile * KB + kb, bar);
                mbar_arrive_expect_tx(bar, W_BYTES + X_BYTES);
            };

            int seg = blockIdx.x;
            long long u0 = seg_begin(p, seg);
            long long u1 = seg_begin(p, seg + 1);
            int tile = (int)(u0 / KB), kb = (int)(u0 % KB);
            // Weights and scales never change between the layers of one stream:
            // prefetch the first stages' weight tiles before waiting for the
            // previous kernel; everything else waits.
            long long pre = 0;
            if (p.early_weights) {
                pre = u1 - u0 < S ? u1 - u0 : S;
                int ptile = tile, pkb = kb;
                for (long long k = 0; k < pre; ++k) {
                    open_stage((int)k, ptile, pkb, seg, k == 0, u1 - u0 - k);
                    issue_w((int)k, ptile, pkb);
                    if (++pkb == KB) { pkb = 0; ++ptile; }
                }
            }
            griddep_wait();
            for (long long k = 0; k < pre; ++k) {
                issue_x((int)k, kb);
                if (++kb == KB) { kb = 0; ++tile; }
            }
            issued = pre;
            long long left = u1 - u0 - pre;
            bool seg_first = pre == 0;
            while (ok) {
                for (; left > 0; --left) {
                    const int s = (int)(issued % S);
                    const uint32_t ph = (uint32_t)((issued / S) & 1);
                    if (issued >= S &&
                        !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, err, kErrProducerWait)) {
                        ok = false;
                        *abort_flag = 1;
                        break;
                    }
                    open_stage(s, tile, kb, seg, seg_first, left);
                    issue_w(s, tile, kb);
                    issue_x(s, kb);
                    seg_first = false;
                    if (++kb == KB) { kb = 0; ++tile; }
                    ++issued;
                }
                if (!ok) break;
                // Claim the next segment after the first wave; the unsigned range
                // check keeps every index in bounds even with a corrupted counter.
                const unsigned claimed = (unsigned)atomicAdd(&p.counter[0], 1);
                if (claimed >= (unsigned)(p.n_segments - G)) break;
                seg = G + (int)claimed;
                u0 = seg_begin(p, seg);
                u1 = seg_begin(p, seg + 1);
                tile = (int)(u0 / KB);
                kb = (int)(u0 % KB);
                left = u1 - u0;
                seg_first = true;
            }
            // Tell the consumers there is no more work.
            {
                const int s = (int)(issued % S);
                const uint32_t ph = (uint32_t)((issued / S) & 1);
                if (issued < S ||
                    mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, err, kErrProducerWait)) {
                    hdr[s].flags = kDone;
                    mbar_arrive(smem_u32(&full[s]));
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
    uint32_t gphase = 0;
    int run_kb0 = 0;
    // Deferred ticket of the last split run (thread 0 only).
    int pend_old = -1, pend_tile = -1, pend_jf = 0, pend_jl = 0;

    // Thread 0 publishes whether the pending split tile is complete; after the
    // barrier every consumer helps finish it.
    auto settle_pending = [&]() -> bool {
        const int fb = (int)(gphase & 1u);
        if (threadIdx.x == 0)
            flag[fb] = (pend_tile >= 0 && pend_old == pend_jl - pend_jf) ? pend_tile : -1;
        if (!group_sync(gbar, gphase, lane, err)) return false;
        const int ft = flag[fb];
        if (ft >= 0) {
            const long long tu0 = (long long)ft * KB;
            fixup_tile<MTB>(p, ft, seg_of(p, tu0), seg_of(p, tu0 + KB - 1), threadIdx.x);
        }
        if (threadIdx.x == 0) {
            if (ft >= 0) p.tickets[ft] = 0;
            pend_tile = -1;
        }
        return true;
    };

    // FP8 MMA: consumer warp w rescales x of token(s) w (and w + 8) of a stage.
    auto prepare_stage = [&](int s) {
        if constexpr (kHalfX) {
            const uint32_t sx = smem_u32(sX + (size_t)s * X_BYTES);
            const uint32_t sxh = smem_u32(sXh + (size_t)s * X_BYTES);
#pragma unroll
            for (int tok = warp; tok < MTB; tok += kConsumerWarps) {
                bool okx = true;
                if (tok < p.M) okx = scale_token_to_f16<MTB>(sx, sxh, tok, lane, unscale + s * 16 + tok);
                if (lane == 0) bad[s * 16 + tok] = okx ? 0 : 1;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&xready[s]));
        }
    };

    bool alive = true;
    if constexpr (kHalfX) {
        // Prologue: prepare stage 0.
        if (!mbar_wait_bounded(smem_u32(&full[0]), 0, err, kErrConsumerWait)) {
            *abort_flag = 1;
            alive = false;
        } else if (!(hdr[0].flags & kDone)) {
            prepare_stage(0);
        }
    }
    for (long long i = 0; alive; ++i) {
        const int s = (int)(i % S);
        const uint32_t ph = (uint32_t)((i / S) & 1);
        if constexpr (!kHalfX) {
            if (!mbar_wait_bounded(smem_u32(&full[s]), ph, err, kErrConsumerWait)) {
                *abort_flag = 1;
                break;
            }
        }
        if (*abort_flag) break;
        const int flags = hdr[s].flags;
        if (flags & kDone) break;
        const int tile = hdr[s].tile, kb = hdr[s].kb;
        const int seg = hdr[s].seg;
        if (flags & kRunFirst) run_kb0 = kb;

        uint32_t sxh = 0;
        const float* uns = nullptr;
        bool exact_bf16 = false;
        if constexpr (kHalfX) {
            // Look one stage ahead: rescale this warp's token of the next stage
            // while the other warps finish this stage's.
            const long long i1 = i + 1;
            const int s1 = (int)(i1 % S);
            if (!mbar_wait_bounded(smem_u32(&full[s1]), (uint32_t)((i1 / S) & 1), err,
                                   kErrConsumerWait)) {
                *abort_flag = 1;
                break;
            }
            if (!(hdr[s1].flags & kDone)) prepare_stage(s1);
            if (!mbar_wait_bounded(smem_u32(&xready[s]), ph, err, kErrConsumerWait)) {
                *abort_flag = 1;
                break;
            }
            sxh = smem_u32(sXh + (size_t)s * X_BYTES);
            uns = unscale + s * 16;
            const uint4 bv = *reinterpret_cast<const uint4*>(bad + s * 16);
            exact_bf16 = ((MTB > 8 ? (bv.z | bv.w) : 0u) | bv.x | bv.y) != 0u;
        }
        float scale = 1.f;
        if constexpr (DT == kFP8) scale = hdr[s].scale;
        c.consume(smem_u32(sW + (size_t)s * W_BYTES), smem_u32(sX + (size_t)s * X_BYTES), sxh, uns,
                  exact_bf16, warp, lane, scale);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        if (flags & kRunLast) {
            // This run of `tile` is complete: store its rows (y, or the slot).
            const bool whole = (run_kb0 == 0) && (kb == KB - 1);
            float* slot = nullptr;
            if (!whole) {
                const long long first_tile = seg_begin(p, seg) / KB;
                slot = p.partials + ((long long)seg * 2 + (tile == first_tile ? 0 : 1)) * MTB * kBN;
            }
            c.write_rows(p, slot, tile * kBN, warp, lane);
            c.reset();
            // Settle the previous split run's ticket (its atomic has had a whole
            // run to complete), then take this one's.
            if (!settle_pending()) { *abort_flag = 1; break; }
            if (!whole && threadIdx.x == 0) {
                const long long tu0 = (long long)tile * KB;
                pend_tile = tile;
                pend_jf = seg_of(p, tu0);
                pend_jl = seg_of(p, tu0 + KB - 1);
                pend_old = atom_add_acq_rel_gpu(&p.tickets[tile], 1);
            }
        }
    }
    // Settle the last pending ticket before leaving.
    if (!*abort_flag) settle_pending();
}

}  // namespace dl
