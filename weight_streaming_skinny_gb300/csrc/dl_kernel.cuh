// The decode-linear kernel: y[M,N] = x[M,K] . w[N,K]^T (+ bias), M <= 16.
//
// Work decomposition ("stream-K").  The weight matrix is cut into tiles of
// kBN = 128 rows; each tile's K range is cut into units of kBK = 128 columns
// (one FP8 scale block).  The U = tiles x k-blocks units, in tile-major order,
// are dealt out as one contiguous range per CTA -- q or q+1 units each -- on a
// persistent grid of about one CTA per SM, so every SM streams the same number
// of weight bytes whatever N and K are.  This is the "split the long dimension
// across blocks so the whole chip streams weights" of "9% faster GLM-5.3-Flash
// prefill with GPU-to-GPU IPC" (section "TileLang: twice as fast, and no
// faster", where a 1..6-token step otherwise launches 16-96 blocks for 188 SMs),
// balanced to one unit.
//
// Pipeline.  Warp 8 (one elected thread) streams units HBM -> shared memory
// with TMA tensor copies into a ring of `stages` buffers, each guarded by a
// full/empty mbarrier pair; the weight tile is 128 rows x 128 bytes per copy
// with the 128-byte swizzle.  Warps 0-7 each own 16 weight rows of the tile
// and consume the ring (the TileLang loop's T.Pipelined(..., num_stages=2),
// deepened to fill GB300's HBM pipe).  Every weight byte is read from HBM
// exactly once per call.
//
// Two consumer families:
//   SIMT: one weight row per lane (two lanes per row, one per K half), CUDA-core
//         fused multiply-adds with bf16 x bf16 -> fp32 products (the row-tiled
//         GEMV of "Developing a custom Qwen2.5 72B inference engine from
//         scratch", §6.1); a shuffle joins the two halves at the end of a tile.
//   MMA:  warp-level mma.sync m16n8k16 bf16 -> fp32 with the weights as the
//         16-row A operand and the (<= 16) tokens as the 8-wide B operand
//         (the "T.gemm(A_s, B_h, acc, transpose_B=True)" of the TileLang loop).
// FP8 weights are decoded exactly e4m3 -> bf16 in registers; the fp32 block
// scale multiplies each 128-wide K block's fp32 partial.
//
// Split-K fix-up.  A tile whose K range lies inside one CTA is finished by it
// (bias, round to bf16, store).  A tile shared by several CTAs: each writes its
// fp32 partial to the workspace, fences, and takes an arrival ticket; the last
// to arrive sums the partials in CTA order (= ascending K), adds the bias,
// rounds once and resets the ticket.  Nobody waits for anybody, and the order
// of every sum is fixed by (M, N, K, grid) alone, so results are bitwise
// reproducible.  Inside one GPU this plays the role of the row-parallel
// "partial sums, then all-reduce" of "Multi-GPU Inference and Serving at
// Scale", Example 3.
#pragma once

#include "dl_device.cuh"

namespace dl {

constexpr int kBN = 128;                 // weight rows per tile
constexpr int kBK = 128;                 // K columns per unit (one FP8 scale block)
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kRedStride = kBN + 4;      // padded row of the per-tile result buffer

enum DType { kBF16 = 0, kFP8 = 1 };
enum Family { kSIMT = 1, kMMA = 2 };

struct LinearParams {
    const uint16_t* bias;     // bf16 [N] or null
    uint16_t* y;              // bf16 [M][N]
    float* y_f32;             // fp32 [M][N] or null
    const float* scales;      // fp32 [ceil(N/128)][KB] (FP8)
    int* tickets;             // [n_tiles] arrival counters (zero between calls)
    float* partials;          // [grid][2][MTB][kBN] fp32
    int M, N, K;
    int KB;                   // k-blocks per tile = ceil(K / 128)
    int n_tiles;
    long long q;              // every CTA gets q units, the first r get one more
    int r;
    int stages;
    unsigned* err;            // device error word (bounded waits OR their bit in)
};

template <int DT>
struct TileBytes {
    static constexpr int w = kBN * kBK * (DT == kBF16 ? 2 : 1);
};

template <int MT>
struct XRows {
    static constexpr int v = MT < 8 ? 8 : MT;   // token rows staged (zero-filled past M)
};

template <int DT, int MT>
__host__ __device__ constexpr int stage_bytes() {
    return TileBytes<DT>::w + XRows<MT>::v * kBK * 2;
}

template <int MT>
__host__ __device__ constexpr int fixed_smem_bytes(int stages) {
    return XRows<MT>::v * kRedStride * 4 + stages * 16 + 16;
}

__device__ __forceinline__ long long unit_begin(int cta, long long q, int r) {
    return (long long)cta * q + (cta < r ? cta : r);
}

// Index of the CTA whose range holds unit u.
__device__ __forceinline__ int cta_of_unit(long long u, long long q, int r) {
    const long long big = (long long)r * (q + 1);
    if (u < big) return (int)(u / (q + 1));
    return r + (int)((u - big) / q);
}

// ------------------------------------------------------------------ consumers

// SIMT consumer.  Lane l of warp w owns weight row 16w + (l & 15) and the K
// half (l >> 4) of every unit: 64 columns = 8 chunks of 16 bytes (bf16) or 4
// chunks (fp8, 16 codes each).  acc[m] is the lane's fp32 sum for token m.
template <int DT, int MT>
struct SimtConsumer {
    static constexpr int MTB = XRows<MT>::v;
    float acc[MT];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    }

    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, int warp, int lane,
                                            float scale) {
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
                    float a = acc[m];
                    a = fma2_bf16(w.x, xv.x, a);
                    a = fma2_bf16(w.y, xv.y, a);
                    a = fma2_bf16(w.z, xv.z, a);
                    a = fma2_bf16(w.w, xv.w, a);
                    acc[m] = a;
                }
            }
        } else {
            const uint32_t wbase = sw + row * 128;
            float part[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) part[m] = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int cc = 4 * h + j;                  // 16-code chunk of the row
                const uint4 w = lds128(wbase + ((cc ^ sw8) << 4));
                uint32_t wb[8];
                wb[0] = e4m3x2_to_bf16x2(w.x & 0xffffu);
                wb[1] = e4m3x2_to_bf16x2(w.x >> 16);
                wb[2] = e4m3x2_to_bf16x2(w.y & 0xffffu);
                wb[3] = e4m3x2_to_bf16x2(w.y >> 16);
                wb[4] = e4m3x2_to_bf16x2(w.z & 0xffffu);
                wb[5] = e4m3x2_to_bf16x2(w.z >> 16);
                wb[6] = e4m3x2_to_bf16x2(w.w & 0xffffu);
                wb[7] = e4m3x2_to_bf16x2(w.w >> 16);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    // codes 16cc..16cc+15 pair with bf16 chunks 2j, 2j+1 of x box h
                    const uint4 x0 = lds128(xbase + m * 128 + (((2 * j) ^ (m & 7)) << 4));
                    const uint4 x1 = lds128(xbase + m * 128 + (((2 * j + 1) ^ (m & 7)) << 4));
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
    }

    // Join the two K halves and write the tile's per-row sums to red[m][row].
    __device__ __forceinline__ void store(float* red, int warp, int lane) {
        const int row = warp * 16 + (lane & 15);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const float other = __shfl_xor_sync(0xffffffffu, acc[m], 16);
            if (lane < 16) red[m * kRedStride + row] = acc[m] + other;
        }
#pragma unroll
        for (int m = MT; m < MTB; ++m)
            if (lane < 16) red[m * kRedStride + row] = 0.f;
    }
};

// MMA consumer.  Warp w owns rows 16w..16w+15 as the A operand of
// mma.m16n8k16; the tokens are the B operand (n = 8, two n-tiles for MT = 16).
// acc[nt][i] follows the mma accumulator layout: thread (g = lane/4,
// t = lane%4) holds rows g and g+8, tokens 8nt + 2t and 8nt + 2t + 1.
template <int DT, int MT>
struct MmaConsumer {
    static_assert(MT == 8 || MT == 16, "MMA consumer stages 8 or 16 tokens");
    static constexpr int NT = MT / 8;
    float acc[NT][4];

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
    }

    __device__ __forceinline__ void consume(uint32_t sw, uint32_t sx, int warp, int lane,
                                            float scale) {
        const int mat = lane >> 3, rr = lane & 7;
        const int arow = warp * 16 + rr + ((mat & 1) << 3);
        const int aswz = arow & 7;
        const uint32_t abase = sw + arow * 128;
        if constexpr (DT == kBF16) {
            // 8 k16 steps; step s reads bf16 chunks 2(s%4), 2(s%4)+1 of box s/4.
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
                    mma_bf16_16816(acc[0], a0[0], a0[1], a0[2], a0[3], b[0], b[1]);
                    mma_bf16_16816(acc[0], a1[0], a1[1], a1[2], a1[3], b[2], b[3]);
                } else {
                    const int tok = rr + ((mat >> 1) << 3);
                    uint32_t b[4], c[4];
                    ldmatrix_x4(xbox + tok * 128 + (((c0 + (mat & 1)) ^ (tok & 7)) << 4),
                                b[0], b[1], b[2], b[3]);
                    ldmatrix_x4(xbox + tok * 128 + (((c0 + 2 + (mat & 1)) ^ (tok & 7)) << 4),
                                c[0], c[1], c[2], c[3]);
                    mma_bf16_16816(acc[0], a0[0], a0[1], a0[2], a0[3], b[0], b[1]);
                    mma_bf16_16816(acc[1], a0[0], a0[1], a0[2], a0[3], b[2], b[3]);
                    mma_bf16_16816(acc[0], a1[0], a1[1], a1[2], a1[3], c[0], c[1]);
                    mma_bf16_16816(acc[1], a1[0], a1[1], a1[2], a1[3], c[2], c[3]);
                }
            }
        } else {
            // 8 k16 steps; step s is the 16-code chunk s of each row.  Thread
            // (g, t) receives codes 4t..4t+3 of its rows' chunk; they stand for
            // fragment columns {2t, 2t+1} and {2t+8, 2t+9}, so its B fragment is
            // x[token][16s + 4t .. 16s + 4t + 3]: 8 bytes of the swizzled x box.
            const int g = lane >> 2, t = lane & 3;
            float part[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) part[nt][i] = 0.f;
#pragma unroll
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
                    const uint32_t xbox = sx + (step >> 2) * (MT * 128);
                    const int xc = 2 * (step & 3) + (t >> 1);      // logical 16-byte chunk
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int tok = g + 8 * nt;
                        const uint2 xb = lds64(xbox + tok * 128 + ((xc ^ (tok & 7)) << 4) + ((t & 1) << 3));
                        mma_bf16_16816(part[nt], A0, A1, A2, A3, xb.x, xb.y);
                    }
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] = fmaf(part[nt][i], scale, acc[nt][i]);
        }
    }

    __device__ __forceinline__ void store(float* red, int warp, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const int row = warp * 16 + g;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int tok = 8 * nt + 2 * t;
            red[tok * kRedStride + row] = acc[nt][0];
            red[(tok + 1) * kRedStride + row] = acc[nt][1];
            red[tok * kRedStride + row + 8] = acc[nt][2];
            red[(tok + 1) * kRedStride + row + 8] = acc[nt][3];
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

// ------------------------------------------------------------------ epilogue

__device__ __forceinline__ void write_output(const LinearParams& p, int m, int n, float v) {
    if (p.bias) v += bf16_bits_to_f32(p.bias[n]);
    const long long o = (long long)m * p.N + n;
    p.y[o] = f32_to_bf16_rne(v);
    if (p.y_f32) p.y_f32[o] = v;
}

// ------------------------------------------------------------------ kernel

template <int DT, int FAM, int MT>
__global__ void __launch_bounds__(kThreads, 1)
linear_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const LinearParams p) {
    using Consumer = typename ConsumerOf<DT, FAM, MT>::type;
    constexpr int MTB = XRows<MT>::v;
    constexpr int W_BYTES = TileBytes<DT>::w;
    constexpr int X_BYTES = MTB * kBK * 2;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int S = p.stages;
    uint8_t* sW = smem;
    uint8_t* sX = sW + (size_t)S * W_BYTES;
    float* red = reinterpret_cast<float*>(sX + (size_t)S * X_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(red + MTB * kRedStride);
    uint64_t* empty = full + S;
    volatile int* flag = reinterpret_cast<volatile int*>(empty + S);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u_begin = unit_begin(cta, p.q, p.r);
    const long long u_end = u_begin + p.q + (cta < p.r ? 1 : 0);
    const int KB = p.KB;
    unsigned* err = p.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        fence_mbarrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tmap(&tm_w);
        prefetch_tmap(&tm_x);
    }
    __syncthreads();

    // ---------------------------------------------------------------- loader
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            long long i = 0;
            for (long long u = u_begin; u < u_end; ++u, ++i) {
                const int s = (int)(i % S);
                const uint32_t ph = (uint32_t)((i / S) & 1);
                if (i >= S &&
                    !mbar_wait_bounded(smem_u32(&empty[s]), ph ^ 1u, err, kErrProducerWait))
                    break;
                const int tile = (int)(u / KB), kb = (int)(u % KB);
                const uint32_t bar = smem_u32(&full[s]);
                const uint32_t dw = smem_u32(sW + (size_t)s * W_BYTES);
                const uint32_t dx = smem_u32(sX + (size_t)s * X_BYTES);
                mbar_arrive_expect_tx(bar, W_BYTES + X_BYTES);
                if constexpr (DT == kBF16) {
                    tma_load_2d(dw, &tm_w, bar, kb * kBK, tile * kBN, pol_w);
                    tma_load_2d(dw + kBN * 128, &tm_w, bar, kb * kBK + 64, tile * kBN, pol_w);
                } else {
                    tma_load_2d(dw, &tm_w, bar, kb * kBK, tile * kBN, pol_w);
                }
                tma_load_2d(dx, &tm_x, bar, kb * kBK, 0, pol_x);
                tma_load_2d(dx + MTB * 128, &tm_x, bar, kb * kBK + 64, 0, pol_x);
            }
            // Do not leave while copies into this CTA's shared memory may be in
            // flight: wait (bounded) for the last phase issued on every stage.
            const long long issued = i;
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
    bool ok = true;
    long long tile_first_u = u_begin;
    const int first_tile = (int)(u_begin / KB);
    long long i = 0;
    for (long long u = u_begin; u < u_end; ++u, ++i) {
        const int s = (int)(i % S);
        const uint32_t ph = (uint32_t)((i / S) & 1);
        const int tile = (int)(u / KB), kb = (int)(u % KB);
        if (ok) ok = mbar_wait_bounded(smem_u32(&full[s]), ph, err, kErrConsumerWait);
        if (ok) {
            float scale = 1.f;
            if constexpr (DT == kFP8) scale = __ldg(p.scales + (long long)tile * KB + kb);
            c.consume(smem_u32(sW + (size_t)s * W_BYTES), smem_u32(sX + (size_t)s * X_BYTES),
                      warp, lane, scale);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        if (kb == KB - 1 || u == u_end - 1) {
            // This CTA's share of `tile` is complete.
            const bool whole = (tile_first_u == (long long)tile * KB) && (kb == KB - 1);
            consumer_sync(kConsumerThreads);           // previous readers of red/flag done
            c.store(red, warp, lane);
            consumer_sync(kConsumerThreads);
            const int n0 = tile * kBN;
            if (whole) {
                for (int idx = threadIdx.x; idx < p.M * kBN; idx += kConsumerThreads) {
                    const int m = idx / kBN, rr = idx % kBN;
                    if (n0 + rr < p.N) write_output(p, m, n0 + rr, red[m * kRedStride + rr]);
                }
            } else {
                const int slot = (tile == first_tile) ? 0 : 1;
                float* mine = p.partials + ((long long)cta * 2 + slot) * MTB * kBN;
                for (int idx = threadIdx.x; idx < p.M * kBN; idx += kConsumerThreads) {
                    const int m = idx / kBN, rr = idx % kBN;
                    mine[idx] = red[m * kRedStride + rr];
                }
                __threadfence();
                consumer_sync(kConsumerThreads);
                const long long tu0 = (long long)tile * KB;
                const int c_first = cta_of_unit(tu0, p.q, p.r);
                const int c_last = cta_of_unit(tu0 + KB - 1, p.q, p.r);
                if (threadIdx.x == 0) {
                    const int old = atomicAdd(&p.tickets[tile], 1);
                    *flag = (old == c_last - c_first) ? 1 : 0;
                }
                consumer_sync(kConsumerThreads);
                if (*flag) {
                    __threadfence();
                    for (int idx = threadIdx.x; idx < p.M * kBN; idx += kConsumerThreads) {
                        const int m = idx / kBN, rr = idx % kBN;
                        if (n0 + rr >= p.N) continue;
                        float v = 0.f;
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            const int cfirst_tile = (int)(unit_begin(cc, p.q, p.r) / KB);
                            const int sl = (tile == cfirst_tile) ? 0 : 1;
                            v += ld_cg_f32(p.partials + (((long long)cc * 2 + sl) * MTB + m) * kBN + rr);
                        }
                        write_output(p, m, n0 + rr, v);
                    }
                    if (threadIdx.x == 0) p.tickets[tile] = 0;
                }
            }
            c.reset();
            tile_first_u = u + 1;
        }
    }
}

}  // namespace dl
