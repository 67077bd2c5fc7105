// C-ABI host side of the decode-linear library: argument validation, the work
// plan (grid, split of K, pipeline depth, workspace layout), TMA descriptor
// encoding, launches, the layer-list stream with optional CUDA-graph replay,
// and error reporting.  Nothing here allocates device memory or synchronises
// the host, except dl_device_status (documented as synchronising).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <list>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "dl_linear.h"
#include "dl_kernel.cuh"
#include "dl_launch.h"

// Device error word: bounded waits in the kernels OR their bit in here.
__device__ unsigned int g_dl_device_error = 0;

// Scratch of dl_linear_bf16_static_scratch: the split-K workspace (counters,
// arrival tickets, partial sums) for callers that cannot allocate one.  One
// copy per device, shared by every call of that entry point.
__device__ __align__(256) unsigned char g_dl_static_scratch[DL_STATIC_SCRATCH_BYTES];

namespace {

thread_local char g_err[512] = "";

dl_status fail(dl_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return s;
}

dl_status ok() {
    g_err[0] = '\0';
    return DL_OK;
}

std::atomic<int> g_kernel_override{0};
std::atomic<int> g_cps_override{0};
std::atomic<int> g_max_ctas_override{0};
// Test hooks of the bounded device waits (dl_set_wait_test): the limit of
// every wait (0: the default) and the stage CTA 0 withholds (0: none).
std::atomic<long long> g_wait_ns_override{0};
std::atomic<int> g_withhold_override{0};

constexpr int kMaxStages = 16;
// bf16 work partition (see make_plan): share of the units in the first wave,
// the smallest later segment in units, and whether later segments are aligned
// to divisors of the units per tile.
constexpr long long kFirstWaveNum = 7, kFirstWaveDen = 8;
// bf16 layers with at most this many units per CTA take FP8's static split
// (same box, two runs each: the bf16 decoder-layer step 0.2691 -> 0.2667 ms,
// gate_up + down at 16 tokens 0.2226 -> 0.2208 ms, one token unchanged; a
// limit of 64 gained less, 32 nothing): a few small claimed segments at the
// end cost such layers more than the balance they buy.
constexpr long long kStaticSplitMaxUnitsPerCta = 128;
constexpr long long kMinSegUnits = 8;
constexpr bool kAlignSegments = true;
// FP8 activation copies made ahead inside a stream go in batches: one launch
// right after every kHoistWindow-th layer (it copies while that layer runs)
// makes the copies of the hoisted layers among the next kHoistWindow.
constexpr int kHoistWindow = 16;
// Stages whose weights a single FP8 call's main kernel fetches while the prep
// kernel runs (more delays its first activation copy).
constexpr int kEarlyStagesAfterPrep = 3;
constexpr int kMaxDevices = 64;
// Workspace prefix that must be zero before a call (and is zero after it):
// the claim/done counters, then one arrival ticket per tile.  Fixed in size,
// so that no call's scratch (partials, FP8 activation copy) ever lies where
// another call's tickets do.
constexpr size_t kTicketsOff = 256;
constexpr int kMaxTiles = 16384;
static_assert(kTicketsOff + (size_t)kMaxTiles * 4 == DL_WORKSPACE_ZERO_BYTES, "zero prefix");
// In the first 256 bytes: int counters [0..3), then the argmax keys (16 x 8 B).
constexpr size_t kArgmaxKeysOff = 64;

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;
    int smem_per_sm = 0;
    unsigned* err_word = nullptr;
};

std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];

dl_status device_info(DeviceInfo& out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(DL_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
            return fail(DL_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_dl_device_error)) != cudaSuccess)
            return fail(DL_ERR_CUDA, "cudaGetSymbolAddress(device error word): %s", cudaGetErrorString(e));
        d.err_word = static_cast<unsigned*>(p);
        d.ready = true;
    }
    out = d;
    return DL_OK;
}

// The work plan of one call: kernel family, staged token rows, tiles, grid
// and the split of the units among CTAs, pipeline depth, workspace layout.
struct Plan {
    int dtype, family, mt, mtb;
    int KB, UT, n_tiles;
    long long units;
    int grid;
    int n_segments;
    int n_waves;
    int wave_seg0[dl::kMaxWaves + 1];
    long long wave_unit0[dl::kMaxWaves];
    int wave_size[dl::kMaxWaves];
    int stages;
    size_t smem;
    size_t counter_off, tickets_off, partials_off, xh_off, unscale_off, ws_bytes;
    size_t xcopy_bytes;       // FP8: the activation copy (f16, or the tensor-memory family's parts)
};

int auto_family(int dtype, int M) {
    // bf16: CUDA-core FMAs at one token, the MMA family from two (same-box
    // bench: gate_up + down at M = 2 run at 0.989 of the copy peak with the
    // MMA family against 0.969 with the CUDA-core one; equal at M = 1).
    if (dtype == DL_BF16) return M <= 1 ? dl::kSIMT : dl::kMMA;
    return dl::kMMA;
}

int pow2_at_least(int M) {
    int t = 1;
    while (t < M) t <<= 1;
    return t;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

dl_status check_shape(int dtype, int M, int N, int K) {
    if (dtype != DL_BF16 && dtype != DL_FP8_B128)
        return fail(DL_ERR_INVALID_ARG, "unknown dtype %d", dtype);
    if (M < 1 || M > 16)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "M=%d outside [1,16] (decode-only skinny GEMM)", M);
    if (N < 1 || K < 1) return fail(DL_ERR_UNSUPPORTED_SHAPE, "N=%d and K=%d must be >= 1", N, K);
    if (dtype == DL_BF16 && K % 8 != 0)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "bf16 weights need K %% 8 == 0 (K=%d)", K);
    if (dtype == DL_FP8_B128 && K % 128 != 0)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "FP8 block-128 weights need K %% 128 == 0 (K=%d)", K);
    return DL_OK;
}

dl_status make_plan(int dtype, int M, int N, int K, const DeviceInfo& di, Plan& pl) {
    pl.dtype = dtype;
    const int ko = g_kernel_override.load();
    pl.family = ko ? ko : auto_family(dtype, M);
    if (pl.family != dl::kSIMT && pl.family != dl::kMMA && pl.family != dl::kTC)
        return fail(DL_ERR_INVALID_ARG, "kernel override %d unknown", pl.family);
    // The tensor-memory family multiplies e4m3 by e4m3: FP8 weights only.
    if (pl.family == dl::kTC && dtype != DL_FP8_B128) pl.family = auto_family(dtype, M);
    // The CUDA-core family decodes FP8 for at most 2 tokens; beyond, the
    // decode cost per code is the same and only the MMA amortises the FMAs.
    if (pl.family == dl::kSIMT && dtype == DL_FP8_B128 && M > 2) pl.family = dl::kMMA;
    pl.mt = pl.family != dl::kSIMT ? (M <= 8 ? 8 : 16) : pow2_at_least(M);
    pl.mtb = dl::host_x_rows(pl.mt);
    pl.KB = (K + dl::kBK - 1) / dl::kBK;
    pl.n_tiles = (N + dl::kBN - 1) / dl::kBN;
    if (pl.n_tiles > kMaxTiles)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "N=%d exceeds %d rows", N, kMaxTiles * dl::kBN);
    // Partition units of 32 KB of weights: one 128-column K block of bf16, two
    // of FP8 (the last one single when KB is odd).
    pl.UT = dtype == DL_BF16 ? pl.KB : (pl.KB + 1) / 2;
    pl.units = (long long)pl.n_tiles * pl.UT;
    // Grid: persistent, `cps` CTAs per SM: by default one, with all of the
    // SM's shared memory; the override ctas_per_sm = 2 sizes the grid for two,
    // each with half of it.
    const int dt_k = dtype == DL_BF16 ? dl::kBF16 : dl::kFP8;
    const int fits = dl::host_min_blocks(dt_k, pl.family, pl.mt);
    const int cps_o = g_cps_override.load();
    int cps = cps_o ? cps_o : fits;
    // Two CTAs per SM stay away from FP8 weights at 16 staged tokens: the one
    // GPU fault ever recorded for this library came from that combination
    // (a build compiled for two resident CTAs, first FP8 16-token call), and
    // reading the code has not explained it.  Such calls keep one CTA per SM.
    if (cps == 2 && dtype == DL_FP8_B128 && pl.mt == 16) cps = 1;
    const bool half_smem = cps == 2;
    long long grid = (long long)di.sm_count * cps;
    const int mc = g_max_ctas_override.load();
    if (mc > 0 && grid > mc) grid = mc;
    if (grid > pl.units) grid = pl.units;
    if (grid < 1) grid = 1;
    pl.grid = (int)grid;
    // Segments: a fixed partition of the units, summed by the fix-up in segment
    // order.  CTA b takes segment b (the first wave, one per CTA).
    //
    // FP8, and bf16 layers of at most kStaticSplitMaxUnitsPerCta units per
    // CTA: that is all -- a static balanced split, U mod G CTAs with one unit
    // more than the others, no segment claimed at run time.  Measured against
    // the bf16 scheme below: FP8 M = 6 layer step 0.1644 -> 0.1544 ms, the
    // 80-layer model 13.13 -> 12.26 ms per token, gate_up + down 0.1298 ->
    // 0.1228 ms (M = 1) and 0.1479 -> 0.1381 ms (M = 16): the small segments of
    // the later waves cost FP8 more in split runs and fix-ups at the end of
    // the call than they gain in balance.  (bf16 is 0.4-1.5 % slower with the
    // static split.)
    //
    // bf16: the first wave holds about 7/8 of the units; then waves of up to
    // `grid` segments, claimed by the CTAs as they finish, each wave covering
    // about half of what is left, down to a minimum size `b`.
    // Every segment that ends inside a tile costs a split run (partial rows,
    // an arrival ticket and, for the last arrival, a fix-up), and those of the
    // last waves land at the end of the call.  So b is large: kMinSegUnits
    // (8 units = 256 KB of weights), at least UT/24 (at most ~24 segments per
    // tile) and M/4 (partial bytes, M x 512 per segment, small next to the
    // segment's weights); if UT is not a multiple of b, a divisor of UT in
    // [b, 2b) is preferred.  When b divides UT, every later wave starts on a
    // multiple of b (an alignment segment of fewer than b units follows the
    // first wave if needed) and holds multiples of b: its segments end on tile
    // boundaries or at multiples of b inside a tile.
    if (dtype == DL_FP8_B128 || pl.units <= (long long)pl.grid * kStaticSplitMaxUnitsPerCta) {
        const long long G = pl.grid, U = pl.units;
        const long long sz = U / G, r = U % G;     // grid <= units, so sz >= 1
        int w = 0;
        if (r > 0) {
            pl.wave_seg0[w] = 0;
            pl.wave_unit0[w] = 0;
            pl.wave_size[w] = (int)(sz + 1);
            ++w;
        }
        pl.wave_seg0[w] = (int)r;
        pl.wave_unit0[w] = r * (sz + 1);
        pl.wave_size[w] = (int)sz;
        ++w;
        pl.n_waves = w;
        pl.n_segments = (int)G;
        pl.wave_seg0[w] = (int)G;
    } else {
        const long long G = pl.grid, U = pl.units, UT = pl.UT;
        long long b = kMinSegUnits;
        const long long by_tile = (UT + 23) / 24;
        const long long by_m = (M + 3) / 4;
        if (by_tile > b) b = by_tile;
        if (by_m > b) b = by_m;
        if (kAlignSegments && UT % b != 0)
            for (long long d = b; d < 2 * b; ++d)
                if (UT % d == 0) {
                    b = d;
                    break;
                }
        const bool aligned = kAlignSegments && UT % b == 0;
        long long s0 = (U * kFirstWaveNum / kFirstWaveDen) / G;
        if (s0 < 1) s0 = 1;
        int w = 0;
        pl.wave_seg0[0] = 0;
        pl.wave_unit0[0] = 0;
        pl.wave_size[0] = (int)s0;
        long long seg = G, unit = G * s0;
        ++w;
        if (aligned && unit < U && unit % b != 0) {
            long long a = b - unit % b;
            if (a > U - unit) a = U - unit;
            pl.wave_seg0[w] = (int)seg;
            pl.wave_unit0[w] = unit;
            pl.wave_size[w] = (int)a;
            seg += 1;
            unit += a;
            ++w;
        }
        while (unit < U) {
            const long long rem = U - unit;
            long long size = rem / (2 * G);
            if (aligned) size -= size % b;
            if (size < b) size = b;
            if (w == dl::kMaxWaves - 1) size = (rem + G - 1) / G;   // last wave takes the rest
            long long count = (rem + size - 1) / size;
            if (count > G) count = G;
            pl.wave_seg0[w] = (int)seg;
            pl.wave_unit0[w] = unit;
            pl.wave_size[w] = (int)size;
            seg += count;
            unit += count * size;
            ++w;
        }
        pl.n_waves = w;
        pl.n_segments = (int)seg;
        pl.wave_seg0[w] = (int)seg;
    }
    // Pipeline depth: as many stages as the shared-memory budget holds.
    int budget = di.smem_optin;
    const int per_sm = (half_smem ? di.smem_per_sm / 2 : di.smem_per_sm) - 1024;
    if (per_sm < budget) budget = per_sm;
    const int dt = dt_k;
    int stages = kMaxStages;
    while (stages > 2 && dl::host_smem_bytes(dt, pl.family, pl.mt, stages) > budget) --stages;
    if (dl::host_smem_bytes(dt, pl.family, pl.mt, stages) > budget)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "not enough shared memory for two pipeline stages");
    pl.stages = stages;
    pl.smem = (size_t)dl::host_smem_bytes(dt, pl.family, pl.mt, stages);
    // Workspace: [claim counter, done counter | pad] [tickets, fixed size]
    // [partials] and for FP8 [f16 copy of x] [unscale factors]; only the
    // first DL_WORKSPACE_ZERO_BYTES must be zero (and are left zero).
    pl.counter_off = 0;
    pl.tickets_off = kTicketsOff;
    pl.partials_off = DL_WORKSPACE_ZERO_BYTES;
    size_t end = pl.partials_off + (size_t)pl.n_segments * 2 * pl.mtb * dl::kBN * sizeof(float);
    pl.xh_off = pl.unscale_off = 0;
    pl.xcopy_bytes = pl.family == dl::kTC ? (size_t)pl.KB * 3 * pl.mtb * 128
                                          : (size_t)pl.KB * 2 * pl.mtb * 64 * 2;
    if (dtype == DL_FP8_B128) {
        pl.xh_off = align_up(end, 256);
        pl.unscale_off = align_up(pl.xh_off + pl.xcopy_bytes, 256);
        end = pl.unscale_off + (size_t)pl.KB * dl::kUnscaleStride * sizeof(float);
    }
    pl.ws_bytes = end;
    return DL_OK;
}

// ----------------------------------------------------------------- TMA descriptors

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

dl_status get_encode(EncodeTiledFn& fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
    });
    if (!g_encode) return fail(DL_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    fn = g_encode;
    return DL_OK;
}

dl_status encode_maps(const Plan& pl, int M, int N, int K, const void* x, const void* W,
                      const float* scales, CUtensorMap& tw, CUtensorMap& tx, CUtensorMap& ts,
                      int& scale_off) {
    EncodeTiledFn enc;
    dl_status s = get_encode(enc);
    if (s != DL_OK) return s;
    const cuuint32_t ones[3] = {1, 1, 1};
    CUresult r;
    if (pl.dtype == DL_BF16) {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)dl::kBN};
        r = enc(&tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(W), dims, strides, box,
                ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K};
        const cuuint32_t box[2] = {128, (cuuint32_t)dl::kBN};
        r = enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box,
                ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(DL_ERR_CUDA, "weight tensor map: CUresult %d", (int)r);
    if (pl.dtype == DL_BF16) {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)pl.mtb};
        r = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), dims, strides, box,
                ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (pl.family == dl::kTC) {
        // The tensor-memory family's e4m3 parts: rows of 128 bytes, [K block]
        // [part][mtb]; one box = the 6 mtb rows of two consecutive K blocks.
        const cuuint64_t dims[2] = {128, (cuuint64_t)pl.KB * 3 * pl.mtb};
        const cuuint64_t strides[1] = {128};
        const cuuint32_t box[2] = {128, (cuuint32_t)(6 * pl.mtb)};
        r = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(x), dims, strides, box,
                ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // The prep kernel's f16 copy: rows of 64 values, [K block][half][mtb];
        // one box = the 4 mtb rows of two consecutive K blocks.
        const cuuint64_t dims[2] = {64, (cuuint64_t)pl.KB * 2 * pl.mtb};
        const cuuint64_t strides[1] = {128};
        const cuuint32_t box[2] = {64, (cuuint32_t)(4 * pl.mtb)};
        r = enc(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(x), dims, strides, box,
                ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return fail(DL_ERR_CUDA, "activation tensor map: CUresult %d", (int)r);
    scale_off = 0;
    if (pl.dtype == DL_BF16) {
        ts = tx;                               // not read by the bf16 kernels
        return DL_OK;
    }
    // The block scales as one row of fp32, from the scales rounded down to 16
    // bytes (the tensor map's base must be; scales need only 4) so that
    // scales[i] is element scale_off + i.  The 16-byte block around scales[0]
    // lies in the same page, allocations begin on 256-byte boundaries, and
    // boxes that run past the last scale read zeros.
    const uintptr_t a = reinterpret_cast<uintptr_t>(scales);
    const uintptr_t base = a & ~static_cast<uintptr_t>(15);
    scale_off = static_cast<int>((a - base) / sizeof(float));
    const cuuint64_t sdims[1] = {(cuuint64_t)scale_off + (cuuint64_t)pl.n_tiles * pl.KB};
    const cuuint64_t sstrides[1] = {0};        // (rank 1: no strides are read)
    const cuuint32_t sbox[1] = {8};
    r = enc(&ts, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, reinterpret_cast<void*>(base), sdims, sstrides,
            sbox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DL_ERR_CUDA, "block-scale tensor map: CUresult %d", (int)r);
    return DL_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host-only checks of one layer (no CUDA call).
dl_status validate(int dtype, int M, int N, int K, const void* x, const void* W,
                   const float* scales, const void* bias, const void* y, const float* y_f32) {
    dl_status s = check_shape(dtype, M, N, K);
    if (s != DL_OK) return s;
    if (!x || !W || !y) return fail(DL_ERR_INVALID_ARG, "x, W and y must be non-NULL");
    if (dtype == DL_FP8_B128 && !scales)
        return fail(DL_ERR_INVALID_ARG, "FP8 block-128 weights need scales");
    if (!aligned(x, 16) || !aligned(W, 16))
        return fail(DL_ERR_MISALIGNED, "x and W must be 16-byte aligned");
    if (!aligned(y, 2) || (bias && !aligned(bias, 2)))
        return fail(DL_ERR_MISALIGNED, "y and bias must be 2-byte aligned");
    if ((y_f32 && !aligned(y_f32, 4)) || (scales && !aligned(scales, 4)))
        return fail(DL_ERR_MISALIGNED, "y_f32 and scales must be 4-byte aligned");
    return DL_OK;
}

dl_status launch_layer(int dtype, int M, int N, int K, const void* x, const void* W,
                       const float* scales, const void* bias, void* y, float* y_f32,
                       void* ws, size_t ws_bytes, cudaStream_t stream, const DeviceInfo& di,
                       bool after_own, int act, int* idx = nullptr, float* maxval = nullptr,
                       uint16_t* xh_ready = nullptr, float* unscale_ready = nullptr,
                       uint16_t* xh_next = nullptr, float* us_next = nullptr,
                       float* wslot = nullptr) {
    // after_own: every earlier kernel on the stream is one of this library's
    // (a later layer of one dl_decode_stream call), so none writes weights or
    // scales and the next one's weights may be fetched before the wait.
    // xh_ready / unscale_ready (FP8): the activation copy was already written
    // there by an earlier launch of the same stream (a prep launch, or the
    // previous layer's epilogue); no prep here.
    // xh_next / us_next / wslot: this layer (act 0, N % 128 == 0) also writes
    // the activation copy of the next layer, an FP8 layer whose x is this y
    // with the same staged token rows; wslot holds grid x 2 slots of
    // [mtb][128] fp32 for the tiles that one segment covers whole.
    Plan pl;
    dl_status s = make_plan(dtype, M, N, K, di, pl);
    if (s != DL_OK) return s;
    if (!ws) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(DL_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    if (ws_bytes < pl.ws_bytes)
        return fail(DL_ERR_WORKSPACE, "workspace has %zu bytes, this call needs %zu", ws_bytes,
                    pl.ws_bytes);
    // FP8: the kernel streams the exact f16 copy of x that the prep kernel
    // writes into the workspace.
    char* wsb = static_cast<char*>(ws);
    uint16_t* xh = dtype == DL_FP8_B128 ? reinterpret_cast<uint16_t*>(wsb + pl.xh_off) : nullptr;
    float* unscale = dtype == DL_FP8_B128 ? reinterpret_cast<float*>(wsb + pl.unscale_off) : nullptr;
    const bool prepped = dtype == DL_FP8_B128 && xh_ready && unscale_ready;
    if (prepped) {
        xh = xh_ready;
        unscale = unscale_ready;
    }
    CUtensorMap tw, tx, ts;
    int scale_off = 0;
    if ((s = encode_maps(pl, M, N, K, xh ? static_cast<const void*>(xh) : x, W, scales, tw, tx, ts,
                         scale_off)) != DL_OK)
        return s;
    dl::LinearParams p;
    p.bias = static_cast<const uint16_t*>(bias);
    p.y = static_cast<uint16_t*>(y);
    p.y_f32 = y_f32;
    p.scales = scales;
    p.scale_off = scale_off;
    p.x = static_cast<const uint16_t*>(x);
    p.unscale = unscale;
    p.counter = reinterpret_cast<int*>(static_cast<char*>(ws) + pl.counter_off);
    p.tickets = reinterpret_cast<int*>(static_cast<char*>(ws) + pl.tickets_off);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + pl.partials_off);
    p.M = M;
    p.N = N;
    p.K = K;
    p.act = act;
    p.ny = act == 1 ? N / 2 : N;
    p.best = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + kArgmaxKeysOff);
    p.idx = idx;
    p.maxval = maxval;
    p.KB = pl.KB;
    p.UT = pl.UT;
    p.n_tiles = pl.n_tiles;
    p.units = pl.units;
    p.n_segments = pl.n_segments;
    p.n_waves = pl.n_waves;
    for (int w = 0; w < dl::kMaxWaves; ++w) {
        p.wave_seg0[w] = w <= pl.n_waves ? pl.wave_seg0[w] : 0;
        p.wave_unit0[w] = w < pl.n_waves ? pl.wave_unit0[w] : 0;
        p.wave_size[w] = w < pl.n_waves ? pl.wave_size[w] : 1;
    }
    p.wave_seg0[dl::kMaxWaves] = pl.wave_seg0[pl.n_waves];
    p.stages = pl.stages;
    p.err = di.err_word;
    const long long wait_o = g_wait_ns_override.load();
    p.wait_ns = wait_o > 0 ? (unsigned long long)wait_o : dl::kWaitLimitNs;
    p.withhold = g_withhold_override.load();
    p.xh_next = xh_next;
    p.us_next = us_next;
    p.wslot = wslot;
    if (xh_next && (act != 0 || N % dl::kBK != 0 || !us_next || !wslot))
        return fail(DL_ERR_INVALID_ARG, "internal: next-layer activation copy needs act 0, "
                    "N %% 128 == 0 and its buffers");
    cudaError_t e;
    if (dtype == DL_BF16) {
        // Inside a stream the previous layer's tail is long: fill the whole ring.
        p.early_stages = after_own ? pl.stages : 0;
        e = dl::launch_linear_bf16(pl.family, pl.mt, tw, tx, p, pl.grid, pl.smem, stream, true);
    } else {
        // The main kernel's attribute first (the only host-side step that can
        // fail for it), then prep -> main.  The prep kernel never writes
        // weights or scales.  Alone, it lets main launch only after its own
        // predecessor has completed, and main then prefetches a few stages
        // during the short prep; inside a stream it lets main launch at once,
        // so main fills its whole ring during the previous layer's tail.
        p.early_stages = after_own ? pl.stages : kEarlyStagesAfterPrep;
        e = dl::launch_linear_fp8(pl.family, pl.mt, tw, tx, ts, p, pl.grid, pl.smem, stream, false);
        if (e == cudaSuccess && !prepped) {
            dl::PrepBatch b{};
            b.n = 1;
            b.layer[0] = dl::PrepLayer{static_cast<const uint16_t*>(x), xh, unscale, M, K, pl.KB, pl.mtb, 0,
                                       pl.family == dl::kTC ? 1 : 0};
            e = dl::launch_prep_x(b, after_own, stream);
        }
        if (e == cudaSuccess)
            e = dl::launch_linear_fp8(pl.family, pl.mt, tw, tx, ts, p, pl.grid, pl.smem, stream, true);
    }
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    return DL_OK;
}

// Raise the shared-memory ceiling of the kernel instance a layer will use
// (host-side, once per device) so that a later stream capture contains only
// launches.
dl_status prepare_layer(int dtype, int M, int N, int K, const DeviceInfo& di) {
    Plan pl;
    dl_status s = make_plan(dtype, M, N, K, di, pl);
    if (s != DL_OK) return s;
    CUtensorMap tw, tx, ts;
    dl::LinearParams p;
    cudaError_t e = dtype == DL_BF16
        ? dl::launch_linear_bf16(pl.family, pl.mt, tw, tx, p, pl.grid, pl.smem, nullptr, false)
        : dl::launch_linear_fp8(pl.family, pl.mt, tw, tx, ts, p, pl.grid, pl.smem, nullptr, false);
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "kernel attribute: %s", cudaGetErrorString(e));
    return DL_OK;
}

// Device address of g_dl_static_scratch on the current device, looked up once
// per device (cudaGetSymbolAddress) and cached.
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

dl_status static_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(DL_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dl_static_scratch);
        if (e != cudaSuccess || !p)
            return fail(DL_ERR_CUDA, "cudaGetSymbolAddress(static scratch): %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return DL_OK;
}

// ----------------------------------------------------------------- stream planning

// Validation of one dl_decode_stream layer (host-only).
dl_status validate_layer(const dl_layer& L, int i) {
    dl_status s = validate(L.dtype, L.M, L.N, L.K, L.x, L.W, L.scales, L.bias, L.y, nullptr);
    if (s == DL_OK && (L.act < 0 || L.act > 2))
        s = fail(DL_ERR_INVALID_ARG, "act %d unknown", L.act);
    if (s == DL_OK && L.act == 2 && !aligned(L.y, 4))
        s = fail(DL_ERR_MISALIGNED, "the argmax indices must be 4-byte aligned");
    if (s == DL_OK && L.act == 1 && L.N % 16 != 0)
        s = fail(DL_ERR_UNSUPPORTED_SHAPE, "SwiGLU needs N %% 16 == 0 (N=%d)", L.N);
    if (s != DL_OK) {
        std::string m = g_err;
        return fail(s, "layer %d: %s", i, m.c_str());
    }
    return DL_OK;
}

// Bytes of y a layer writes (bf16 [M][N or N/2], or int32 [M] indices).
size_t y_bytes(const dl_layer& L) {
    if (L.act == 2) return (size_t)4 * L.M;
    return (size_t)2 * L.M * (L.act == 1 ? L.N / 2 : L.N);
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

// The workspace the layers need one at a time (the largest single plan), and
// where the FP8 layers whose activations are ready when the stream starts --
// no earlier layer of the stream writes any byte of their x -- keep their f16
// copies: one region each after that, so that the copies are made ahead (in
// batches placed every kHoistWindow layers) and those layers then follow one
// another like bf16 layers.  `limit` = the caller's workspace (0: no limit);
// layers that do not fit get their own prep launch as usual.  off[i] = 0: not
// hoisted.
// Then the FP8 layers fed by the layer just before them -- x is exactly that
// layer's whole y, a plain linear (act 0) with the same M and staged token
// rows -- get their copy from that layer's epilogue instead of a prep launch
// (fed[i] = its region, 0: none).  The copies of such layers alternate
// between two regions, so that a layer never writes the copy it reads; the
// producing layers share one set of per-CTA slots at `wslot`.
dl_status plan_stream(const dl_layer* layers, int n, const DeviceInfo& di, size_t limit,
                      size_t& base, std::vector<size_t>& off, size_t& end,
                      std::vector<size_t>& fed, size_t& wslot) {
    base = 0;
    for (int i = 0; i < n; ++i) {
        Plan pl;
        dl_status s = make_plan(layers[i].dtype, layers[i].M, layers[i].N, layers[i].K, di, pl);
        if (s != DL_OK) return s;
        base = pl.ws_bytes > base ? pl.ws_bytes : base;
    }
    off.assign((size_t)n, 0);
    end = align_up(base, 256);
    for (int i = 0; i < n; ++i) {
        const dl_layer& L = layers[i];
        if (L.dtype != DL_FP8_B128) continue;
        bool ready = true;
        const size_t xb = (size_t)2 * L.M * L.K;
        for (int j = 0; j < i && ready; ++j) ready = !overlaps(L.x, xb, layers[j].y, y_bytes(layers[j]));
        if (!ready) continue;
        Plan pl;
        dl_status s = make_plan(L.dtype, L.M, L.N, L.K, di, pl);
        if (s != DL_OK) return s;
        const size_t need = align_up(pl.xcopy_bytes, 256) +
                            align_up((size_t)pl.KB * dl::kUnscaleStride * sizeof(float), 256);
        if (limit && end + need > limit) continue;
        off[(size_t)i] = end;
        end += need;
    }
    fed.assign((size_t)n, 0);
    wslot = 0;
    size_t region = 0, slots = 0;       // the largest copy and the largest slot set
    std::vector<char> is_fed((size_t)n, 0);
    for (int i = 1; i < n; ++i) {
        const dl_layer& L = layers[i];
        const dl_layer& P = layers[i - 1];
        if (L.dtype != DL_FP8_B128 || off[(size_t)i] || P.act != 0) continue;
        if (L.x != P.y || L.M != P.M || L.K != P.N) continue;
        Plan pl, pp;
        dl_status s = make_plan(L.dtype, L.M, L.N, L.K, di, pl);
        if (s == DL_OK) s = make_plan(P.dtype, P.M, P.N, P.K, di, pp);
        if (s != DL_OK) return s;
        // the epilogue writes the f16 copy (not the tensor-memory family's parts)
        if (pp.mtb != pl.mtb || pl.family == dl::kTC) continue;
        const size_t need = align_up(pl.xcopy_bytes, 256) +
                            align_up((size_t)pl.KB * dl::kUnscaleStride * sizeof(float), 256);
        const size_t sl = align_up((size_t)pp.grid * 2 * pp.mtb * dl::kBN * sizeof(float), 256);
        const size_t r = need > region ? need : region, w = sl > slots ? sl : slots;
        if (limit && end + 2 * r + w > limit) continue;
        region = r;
        slots = w;
        is_fed[(size_t)i] = 1;
    }
    if (region) {
        const size_t r0 = end, r1 = end + region;
        wslot = end + 2 * region;
        end = wslot + slots;
        int k = 0;
        for (int i = 1; i < n; ++i)
            if (is_fed[(size_t)i]) fed[(size_t)i] = (k++ & 1) ? r1 : r0;
    }
    return DL_OK;
}

// ----------------------------------------------------------------- graph cache

// Cached executable graphs of dl_decode_stream, least recently used first
// out.  The key is built from the layers' fields (never from the struct's
// raw bytes, whose padding a C caller may leave uninitialised).
constexpr size_t kGraphCacheSize = 16;
std::mutex g_graph_mu;
std::list<std::pair<std::string, cudaGraphExec_t>> g_graph_lru;   // most recent first
std::map<std::string, std::list<std::pair<std::string, cudaGraphExec_t>>::iterator> g_graphs;

std::string graph_key(const dl_layer* layers, int n, const void* ws, size_t ws_bytes, int dev) {
    std::vector<long long> k;
    k.reserve((size_t)n * 10 + 10);
    for (int i = 0; i < n; ++i) {
        const dl_layer& L = layers[i];
        k.insert(k.end(), {(long long)L.dtype, (long long)L.M, (long long)L.N, (long long)L.K,
                           (long long)L.act, (long long)(uintptr_t)L.x, (long long)(uintptr_t)L.W,
                           (long long)(uintptr_t)L.scales, (long long)(uintptr_t)L.bias,
                           (long long)(uintptr_t)L.y});
    }
    k.insert(k.end(), {(long long)(uintptr_t)ws, (long long)ws_bytes, (long long)dev,
                       (long long)g_kernel_override.load(), (long long)g_cps_override.load(),
                       (long long)g_max_ctas_override.load(), g_wait_ns_override.load(),
                       (long long)g_withhold_override.load()});
    return std::string(reinterpret_cast<const char*>(k.data()), k.size() * sizeof(long long));
}

}  // namespace

extern "C" {

int dl_version(void) { return DL_VERSION; }

const char* dl_last_error(void) { return g_err; }

dl_status dl_set_override(int kernel, int ctas_per_sm, int max_ctas) {
    if (kernel < 0 || kernel > 3) return fail(DL_ERR_INVALID_ARG, "kernel override %d unknown", kernel);
    if (ctas_per_sm < 0 || ctas_per_sm > 2)
        return fail(DL_ERR_INVALID_ARG, "ctas_per_sm must be 0, 1 or 2");
    if (max_ctas < 0) return fail(DL_ERR_INVALID_ARG, "max_ctas must be >= 0");
    g_kernel_override.store(kernel);
    g_cps_override.store(ctas_per_sm);
    g_max_ctas_override.store(max_ctas);
    return ok();
}

size_t dl_workspace_bytes(int M, int N, int K, int dtype) {
    if (check_shape(dtype, M, N, K) != DL_OK) return 0;
    DeviceInfo di;
    if (device_info(di) != DL_OK) return 0;
    Plan pl;
    if (make_plan(dtype, M, N, K, di, pl) != DL_OK) return 0;
    return pl.ws_bytes;
}

dl_status dl_linear_bf16(const void* x, const void* W, const void* bias, void* y, float* y_f32,
                         int M, int N, int K, void* workspace, size_t ws_bytes, void* stream) {
    dl_status s = validate(DL_BF16, M, N, K, x, W, nullptr, bias, y, y_f32);
    if (s != DL_OK) return s;
    if (!workspace) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    DeviceInfo di;
    if ((s = device_info(di)) != DL_OK) return s;
    s = launch_layer(DL_BF16, M, N, K, x, W, nullptr, bias, y, y_f32, workspace, ws_bytes,
                     static_cast<cudaStream_t>(stream), di, false, 0);
    return s == DL_OK ? ok() : s;
}

dl_status dl_linear_bf16_static_scratch(const void* x, const void* W, const void* bias, void* y,
                                        float* y_f32, int M, int N, int K, void* stream) {
    dl_status s = validate(DL_BF16, M, N, K, x, W, nullptr, bias, y, y_f32);
    if (s != DL_OK) return s;
    DeviceInfo di;
    if ((s = device_info(di)) != DL_OK) return s;
    Plan pl;
    if ((s = make_plan(DL_BF16, M, N, K, di, pl)) != DL_OK) return s;
    if (pl.ws_bytes > (size_t)DL_STATIC_SCRATCH_BYTES)
        return fail(DL_ERR_WORKSPACE,
                    "M=%d N=%d K=%d needs %zu bytes of scratch; the static scratch holds %zu "
                    "(use dl_linear_bf16 with a workspace)",
                    M, N, K, pl.ws_bytes, (size_t)DL_STATIC_SCRATCH_BYTES);
    void* scratch = nullptr;
    if ((s = static_scratch(&scratch)) != DL_OK) return s;
    // The claim/done counters and the arrival tickets must start at zero; the
    // partial slots are always written before they are read.
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, pl.tickets_off + (size_t)pl.n_tiles * sizeof(int), st);
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "clearing the static scratch: %s", cudaGetErrorString(e));
    s = launch_layer(DL_BF16, M, N, K, x, W, nullptr, bias, y, y_f32, scratch,
                     (size_t)DL_STATIC_SCRATCH_BYTES, st, di, false, 0);
    return s == DL_OK ? ok() : s;
}

dl_status dl_linear_fp8_block128(const void* x, const void* Wq, const float* scales,
                                 const void* bias, void* y, float* y_f32, int M, int N, int K,
                                 void* workspace, size_t ws_bytes, void* stream) {
    dl_status s = validate(DL_FP8_B128, M, N, K, x, Wq, scales, bias, y, y_f32);
    if (s != DL_OK) return s;
    if (!workspace) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    DeviceInfo di;
    if ((s = device_info(di)) != DL_OK) return s;
    s = launch_layer(DL_FP8_B128, M, N, K, x, Wq, scales, bias, y, y_f32, workspace, ws_bytes,
                     static_cast<cudaStream_t>(stream), di, false, 0);
    return s == DL_OK ? ok() : s;
}

dl_status dl_linear_argmax(int dtype, const void* x, const void* W, const float* scales,
                           const void* bias, int* idx, float* maxval, void* y, float* y_f32, int M,
                           int N, int K, void* workspace, size_t ws_bytes, void* stream) {
    if (dtype != DL_BF16 && dtype != DL_FP8_B128)
        return fail(DL_ERR_INVALID_ARG, "dtype %d unknown", dtype);
    if (!idx) return fail(DL_ERR_INVALID_ARG, "idx must be non-NULL");
    if (!aligned(idx, 4) || (maxval && !aligned(maxval, 4)))
        return fail(DL_ERR_MISALIGNED, "idx and maxval must be 4-byte aligned");
    // y is optional here: validate with a stand-in when it is absent.
    dl_status s = validate(dtype, M, N, K, x, W, scales, bias, y ? y : static_cast<void*>(idx), y_f32);
    if (s != DL_OK) return s;
    if (!workspace) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    DeviceInfo di;
    if ((s = device_info(di)) != DL_OK) return s;
    s = launch_layer(dtype, M, N, K, x, W, scales, bias, y, y_f32, workspace, ws_bytes,
                     static_cast<cudaStream_t>(stream), di, false, 2, idx, maxval);
    return s == DL_OK ? ok() : s;
}

dl_status dl_linear_swiglu(int dtype, const void* x, const void* W, const float* scales,
                           const void* bias, void* y, float* y_f32, int M, int N, int K,
                           void* workspace, size_t ws_bytes, void* stream) {
    if (dtype != DL_BF16 && dtype != DL_FP8_B128)
        return fail(DL_ERR_INVALID_ARG, "dtype %d unknown", dtype);
    dl_status s = validate(dtype, M, N, K, x, W, scales, bias, y, y_f32);
    if (s != DL_OK) return s;
    if (N % 16 != 0)
        return fail(DL_ERR_UNSUPPORTED_SHAPE, "SwiGLU needs N %% 16 == 0 (N=%d)", N);
    if (!workspace) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    DeviceInfo di;
    if ((s = device_info(di)) != DL_OK) return s;
    s = launch_layer(dtype, M, N, K, x, W, scales, bias, y, y_f32, workspace, ws_bytes,
                     static_cast<cudaStream_t>(stream), di, false, 1);
    return s == DL_OK ? ok() : s;
}

dl_status dl_decode_stream(const dl_layer* layers, int n_layers, void* workspace, size_t ws_bytes,
                           void* stream, int use_graph) {
    if (n_layers < 0 || (n_layers > 0 && !layers))
        return fail(DL_ERR_INVALID_ARG, "layers must be non-NULL when n_layers > 0");
    if (use_graph != 0 && use_graph != 1) return fail(DL_ERR_INVALID_ARG, "use_graph must be 0 or 1");
    for (int i = 0; i < n_layers; ++i) {
        dl_status s = validate_layer(layers[i], i);
        if (s != DL_OK) return s;
    }
    if (n_layers == 0) return ok();
    if (!workspace) return fail(DL_ERR_WORKSPACE, "workspace is NULL");
    DeviceInfo di;
    dl_status s = device_info(di);
    if (s != DL_OK) return s;
    // Check every layer's plan against the workspace before enqueuing anything.
    for (int i = 0; i < n_layers; ++i) {
        const dl_layer& L = layers[i];
        Plan pl;
        if ((s = make_plan(L.dtype, L.M, L.N, L.K, di, pl)) != DL_OK) return s;
        if (ws_bytes < pl.ws_bytes)
            return fail(DL_ERR_WORKSPACE, "layer %d needs %zu workspace bytes, have %zu", i,
                        pl.ws_bytes, ws_bytes);
        if ((s = prepare_layer(L.dtype, L.M, L.N, L.K, di)) != DL_OK) return s;
    }
    size_t base = 0, end = 0, wslot = 0;
    std::vector<size_t> hoist, fed;
    if ((s = plan_stream(layers, n_layers, di, ws_bytes, base, hoist, end, fed, wslot)) != DL_OK) return s;
    char* wsb = static_cast<char*>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto enqueue_all = [&]() -> dl_status {
        // The activation copies of the FP8 layers whose x is ready at the
        // start (hoist[i] != 0): layer 0's alone before it (it waits for the
        // kernels before the stream, and only then lets layer 0 launch); every
        // later one's in launches of up to kMaxPrepLayers placed right after
        // layer 0's kernel, which copy while it runs and complete only after
        // it (wait_last).
        bool any = false;
        auto region = [&](int i, const Plan& pl, uint16_t*& xh, float*& us) {
            const size_t o = hoist[(size_t)i] ? hoist[(size_t)i] : fed[(size_t)i];
            xh = reinterpret_cast<uint16_t*>(wsb + o);
            us = reinterpret_cast<float*>(wsb + o + align_up(pl.xcopy_bytes, 256));
        };
        auto enqueue_copies = [&](int from, int to, bool wait_last) -> dl_status {
            dl::PrepBatch b{};
            b.wait_last = wait_last ? 1 : 0;
            for (int i = from; i < to; ++i) {
                if (!hoist[(size_t)i]) continue;
                const dl_layer& L = layers[i];
                Plan pl;
                dl_status r = make_plan(L.dtype, L.M, L.N, L.K, di, pl);
                if (r != DL_OK) return r;
                uint16_t* xh;
                float* us;
                region(i, pl, xh, us);
                b.layer[b.n++] = dl::PrepLayer{static_cast<const uint16_t*>(L.x), xh, us, L.M, L.K, pl.KB,
                                               pl.mtb, 0, pl.family == dl::kTC ? 1 : 0};
                if (b.n == dl::kMaxPrepLayers || i == to - 1) {
                    const cudaError_t e = dl::launch_prep_x(b, false, st);
                    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "prep launch: %s", cudaGetErrorString(e));
                    any = true;
                    b.n = 0;
                }
            }
            if (b.n) {
                const cudaError_t e = dl::launch_prep_x(b, false, st);
                if (e != cudaSuccess) return fail(DL_ERR_CUDA, "prep launch: %s", cudaGetErrorString(e));
                any = true;
            }
            return DL_OK;
        };
        // Layer 0's copy goes alone before it; the copies of the hoisted
        // layers in (16k, 16k + 16] go in a batch right after layer 16k, which
        // copies while that layer runs.  If layer 0 has no copy of its own
        // made here, its kernel may let the next one start before the kernels
        // before the stream are done: the first window's copies then go
        // before it, waiting first.
        const bool split = hoist[0] != 0;
        dl_status r0 = enqueue_copies(0, split ? 1 : (n_layers < kHoistWindow + 1 ? n_layers : kHoistWindow + 1),
                                      false);
        if (r0 != DL_OK) return r0;
        for (int i = 0; i < n_layers; ++i) {
            const dl_layer& L = layers[i];
            // Layers after the first, or after a prep launch, follow one of this
            // library's own kernels, which never writes weights: they may
            // prefetch their first weight tiles while that kernel drains.
            const bool after_own = i > 0 || any;
            uint16_t* xh = nullptr;
            float* us = nullptr;
            if (hoist[(size_t)i] || fed[(size_t)i]) {
                Plan pl;
                dl_status r = make_plan(L.dtype, L.M, L.N, L.K, di, pl);
                if (r != DL_OK) return r;
                region(i, pl, xh, us);
            }
            // The next layer's copy, when this layer's epilogue makes it.
            uint16_t* xh_next = nullptr;
            float* us_next = nullptr;
            float* slots = nullptr;
            if (i + 1 < n_layers && fed[(size_t)i + 1]) {
                const dl_layer& Q = layers[i + 1];
                Plan pq;
                dl_status r = make_plan(Q.dtype, Q.M, Q.N, Q.K, di, pq);
                if (r != DL_OK) return r;
                region(i + 1, pq, xh_next, us_next);
                slots = reinterpret_cast<float*>(wsb + wslot);
            }
            // act = 2: y holds the int32 argmax indices; no logits are written.
            dl_status r = L.act == 2
                ? launch_layer(L.dtype, L.M, L.N, L.K, L.x, L.W, L.scales, L.bias, nullptr, nullptr,
                               workspace, ws_bytes, st, di, after_own, 2, static_cast<int*>(L.y),
                               nullptr, xh, us)
                : launch_layer(L.dtype, L.M, L.N, L.K, L.x, L.W, L.scales, L.bias, L.y, nullptr,
                               workspace, ws_bytes, st, di, after_own, L.act, nullptr, nullptr, xh, us,
                               xh_next, us_next, slots);
            if (r != DL_OK) {
                std::string m = g_err;
                return fail(r, "layer %d: %s", i, m.c_str());
            }
            if (i % kHoistWindow == 0 && (i > 0 || split)) {
                const int to = i + kHoistWindow + 1 < n_layers ? i + kHoistWindow + 1 : n_layers;
                if ((r = enqueue_copies(i + 1, to, true)) != DL_OK) return r;
            }
        }
        return DL_OK;
    };
    if (!use_graph) {
        s = enqueue_all();
        return s == DL_OK ? ok() : s;
    }
    if (st == nullptr)
        return fail(DL_ERR_INVALID_ARG, "graph replay needs a non-default stream");
    int dev = 0;
    cudaGetDevice(&dev);
    const std::string key = graph_key(layers, n_layers, workspace, ws_bytes, dev);
    cudaGraphExec_t exec = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_graph_mu);
        auto it = g_graphs.find(key);
        if (it != g_graphs.end()) {
            g_graph_lru.splice(g_graph_lru.begin(), g_graph_lru, it->second);   // now most recent
            exec = it->second->second;
        }
    }
    cudaError_t e;
    if (!exec) {
        if ((e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal)) != cudaSuccess)
            return fail(DL_ERR_CUDA, "cudaStreamBeginCapture: %s", cudaGetErrorString(e));
        dl_status r = enqueue_all();
        cudaGraph_t graph = nullptr;
        e = cudaStreamEndCapture(st, &graph);
        if (r != DL_OK) {
            if (graph) cudaGraphDestroy(graph);
            return r;
        }
        if (e != cudaSuccess) return fail(DL_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return fail(DL_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(e));
        std::lock_guard<std::mutex> lk(g_graph_mu);
        auto it = g_graphs.find(key);
        if (it != g_graphs.end()) {            // another thread cached the same list meanwhile
            cudaGraphExecDestroy(it->second->second);
            it->second->second = exec;
            g_graph_lru.splice(g_graph_lru.begin(), g_graph_lru, it->second);
        } else {
            if (g_graph_lru.size() >= kGraphCacheSize) {
                // A graph still in flight is freed once its launches complete.
                cudaGraphExecDestroy(g_graph_lru.back().second);
                g_graphs.erase(g_graph_lru.back().first);
                g_graph_lru.pop_back();
            }
            g_graph_lru.emplace_front(key, exec);
            g_graphs[key] = g_graph_lru.begin();
        }
    }
    if ((e = cudaGraphLaunch(exec, st)) != cudaSuccess)
        return fail(DL_ERR_CUDA, "cudaGraphLaunch: %s", cudaGetErrorString(e));
    return ok();
}

size_t dl_decode_stream_workspace_bytes(const dl_layer* layers, int n_layers) {
    if (n_layers <= 0 || !layers) return 0;
    for (int i = 0; i < n_layers; ++i)
        if (validate_layer(layers[i], i) != DL_OK) return 0;
    DeviceInfo di;
    if (device_info(di) != DL_OK) return 0;
    size_t base = 0, end = 0, wslot = 0;
    std::vector<size_t> hoist, fed;
    if (plan_stream(layers, n_layers, di, 0, base, hoist, end, fed, wslot) != DL_OK) return 0;
    return end > base ? end : base;
}

int dl_decode_stream_launches(const dl_layer* layers, int n_layers, size_t ws_bytes) {
    if (n_layers < 0 || (n_layers > 0 && !layers)) return -1;
    if (n_layers == 0) return 0;
    for (int i = 0; i < n_layers; ++i)
        if (validate_layer(layers[i], i) != DL_OK) return -1;
    DeviceInfo di;
    if (device_info(di) != DL_OK) return -1;
    size_t base = 0, end = 0, wslot = 0;
    std::vector<size_t> hoist, fed;
    if (plan_stream(layers, n_layers, di, ws_bytes, base, hoist, end, fed, wslot) != DL_OK) return -1;
    int hoisted = 0, fp8 = 0, by_epilogue = 0, batches = 0;
    for (int i = 0; i < n_layers; ++i) {
        fp8 += layers[i].dtype == DL_FP8_B128;
        hoisted += hoist[(size_t)i] != 0;
        by_epilogue += fed[(size_t)i] != 0;
    }
    // the batches of copies made ahead, window by window as enqueued: the
    // first window before layer 0 when layer 0 has no copy of its own, else
    // layer 0's alone before it and each window after its first layer
    const bool split = hoist[0] != 0;
    auto count = [&](int from, int to) {
        int c = 0;
        for (int i = from; i < to; ++i) c += hoist[(size_t)i] != 0;
        return (c + dl::kMaxPrepLayers - 1) / dl::kMaxPrepLayers;
    };
    batches += count(0, split ? 1 : (n_layers < kHoistWindow + 1 ? n_layers : kHoistWindow + 1));
    for (int i = 0; i < n_layers; i += kHoistWindow)
        if (i > 0 || split) batches += count(i + 1, i + kHoistWindow + 1 < n_layers ? i + kHoistWindow + 1 : n_layers);
    // one main kernel per layer, and a prep kernel before every other FP8
    // layer whose copy the layer before does not make
    return batches + n_layers + (fp8 - hoisted - by_epilogue);
}

void dl_graph_cache_clear(void) {
    std::lock_guard<std::mutex> lk(g_graph_mu);
    for (auto& kv : g_graph_lru) cudaGraphExecDestroy(kv.second);
    g_graph_lru.clear();
    g_graphs.clear();
}

int dl_graph_cache_size(void) {
    std::lock_guard<std::mutex> lk(g_graph_mu);
    return (int)g_graph_lru.size();
}

dl_status dl_set_wait_test(long long wait_limit_ns, int withhold_stage) {
    if (wait_limit_ns < 0) return fail(DL_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
    if (withhold_stage < 0) return fail(DL_ERR_INVALID_ARG, "withhold_stage must be >= 0");
    if (withhold_stage > 0 && (wait_limit_ns <= 0 || wait_limit_ns > 100000000LL))
        return fail(DL_ERR_INVALID_ARG,
                    "withholding a stage needs a wait limit in (0, 100 ms] (got %lld ns)", wait_limit_ns);
    g_wait_ns_override.store(wait_limit_ns);
    g_withhold_override.store(withhold_stage);
    return ok();
}

dl_status dl_device_status(unsigned int* flags) {
    unsigned v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(DL_ERR_CUDA, "cudaDeviceSynchronize: %s", cudaGetErrorString(e));
    if ((e = cudaMemcpyFromSymbol(&v, g_dl_device_error, sizeof v)) != cudaSuccess)
        return fail(DL_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
    const unsigned zero = 0;
    if ((e = cudaMemcpyToSymbol(g_dl_device_error, &zero, sizeof zero)) != cudaSuccess)
        return fail(DL_ERR_CUDA, "clearing the device error word: %s", cudaGetErrorString(e));
    if (flags) *flags = v;
    if (v) return fail(DL_ERR_DEVICE, "device error word 0x%x (a bounded wait gave up)", v);
    return ok();
}

}  // extern "C"
