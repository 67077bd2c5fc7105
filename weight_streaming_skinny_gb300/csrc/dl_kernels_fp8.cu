// FP8 (e4m3, 128x128 block scales) instances of the decode-linear kernel.
#include "dl_kernels_common.cuh"

namespace dl {

// ------------------------------------------------------------------ FP8 activation prep

// x (bf16 [M][K]) -> xh (f16): each (token, 128-column block) is scaled
// by 2^(141 - e), e the largest biased exponent of the block's values, so that
// its largest magnitude lands in [2^14, 2^15); every value is then exact in
// f16 if no non-zero value has a biased exponent below e - 31 (f16 subnormals
// keep 8 significant bits down to 2^-17) and none is an infinity or NaN.
// unscale[kb][tok] = 2^(e - 141) (1 for an all-zero block and for the token
// slots tok >= M), or 0 when the block is not exact in f16.  xh is laid out
// [K block][half][mtb token rows][64], rows tok >= M zero, so that the main
// kernel fetches the activations of one or two K blocks with one tensor copy.
// Within every group of 16 columns the values are stored in the order the
// FP8 MMA fragments take them (position 2t + j holds column 4t + j and
// position 2t + 8 + j holds column 4t + 2 + j, t < 4, j < 2): a plain
// ldmatrix of a token row then yields the B fragment that matches the e4m3
// codes 4t .. 4t + 3 a thread receives for the A operand.
// One warp per (block, token slot); lane l handles 4 values.  K % 128 == 0.
__global__ void __launch_bounds__(256) prep_x_kernel(const uint16_t* __restrict__ x,
                                                     uint16_t* __restrict__ xh,
                                                     float* __restrict__ unscale, int M, int K,
                                                     int KB, int mtb, int early_trigger) {
    // x may be the previous kernel's output: wait for it.  The main kernel that
    // follows prefetches weights as soon as this grid lets it launch, so unless
    // every kernel before is known never to write weights (early_trigger, inside
    // one decode stream) it is let launch only after that wait.
    if (early_trigger) griddep_launch_dependents();
    griddep_wait();
    if (!early_trigger) griddep_launch_dependents();
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int kb = w / kUnscaleStride, tok = w % kUnscaleStride;
    if (kb >= KB) return;
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
    const uint2 v = ldg64(x + (long long)tok * K + (long long)kb * kBK + lane * 4);
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


cudaError_t launch_linear_fp8(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                              const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                              bool launch) {
    return launch_family<kFP8>(family, mt, tw, tx, p, grid, smem, stream, launch);
}

cudaError_t launch_prep_x(const uint16_t* x, uint16_t* xh, float* unscale, int M, int K, int KB,
                          int mtb, bool early_trigger, cudaStream_t stream) {
    // One warp per (k-block, token slot), 8 warps per block.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((KB * kUnscaleStride + 7) / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e =
        cudaLaunchKernelEx(&cfg, prep_x_kernel, x, xh, unscale, M, K, KB, mtb, early_trigger ? 1 : 0);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dl
