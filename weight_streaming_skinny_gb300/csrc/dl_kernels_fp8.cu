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
// One launch covers up to kMaxPrepLayers layers (blockIdx.y = layer): the
// copies of every layer of a decode stream whose x is ready when the stream
// starts.
// The four x values lane `lane` of a pair's warp converts (zero for the token
// slots >= M).
__device__ __forceinline__ uint2 load_pair(const PrepLayer& L, int kb, int tok, int lane) {
    if (tok >= L.M) return make_uint2(0u, 0u);
    return ldg64(L.x + (long long)tok * L.K + (long long)kb * kBK + lane * 4);
}

// One pair: this warp's (K block, token slot) of layer L, from its values v.
__device__ __forceinline__ void prep_pair(const PrepLayer& L, int kb, int tok, int lane, uint2 v) {
    if (L.parts)
        write_x_parts_pair(reinterpret_cast<uint8_t*>(L.xh), L.unscale, L.M, L.mtb, kb, tok, lane, v);
    else
        write_x_copy_pair(L.xh, L.unscale, L.M, L.mtb, kb, tok, lane, v);
}

template <int NB>
__global__ void __launch_bounds__(256) prep_x_kernel(const __grid_constant__ PrepBatchN<NB> batch) {
    const int lane = threadIdx.x & 31;
    // (copies made ahead always use the batched instance, NB > 1, even for one
    // layer: that code is left out of the single-layer one)
    if (NB > 1 && batch.wait_last) {
        // x is ready already (see PrepBatch): copy it while the previous
        // kernel runs, then complete only after that kernel has (every thread
        // waits), so that a kernel waiting for this grid also waits for it.
        // A small grid (at most one block per SM) walks all layers' pairs,
        // kPrepInFlight loads in flight per warp, so that its waiting blocks
        // leave room for the next kernel's CTAs.
        griddep_launch_dependents();
        const int nw = gridDim.x * 8, w0 = blockIdx.x * 8 + (threadIdx.x >> 5);
        const int total = batch.layer[batch.n - 1].pair0 + batch.layer[batch.n - 1].KB * kUnscaleStride;
        for (int q0 = w0; q0 < total; q0 += nw * kPrepInFlight) {
            uint2 v[kPrepInFlight];
            int li[kPrepInFlight];
#pragma unroll
            for (int i = 0; i < kPrepInFlight; ++i) {
                const int q = q0 + i * nw;
                int l = 0;
                while (l + 1 < batch.n && batch.layer[l + 1].pair0 <= q) ++l;
                li[i] = l;
                const int r = q - batch.layer[l].pair0;
                v[i] = q < total ? load_pair(batch.layer[l], r / kUnscaleStride, r % kUnscaleStride, lane)
                                 : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < kPrepInFlight; ++i) {
                const int q = q0 + i * nw;
                if (q >= total) break;
                const int r = q - batch.layer[li[i]].pair0;
                prep_pair(batch.layer[li[i]], r / kUnscaleStride, r % kUnscaleStride, lane, v[i]);
            }
        }
        griddep_wait();
        return;
    }
    const int w = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int kb = w / kUnscaleStride, tok = w % kUnscaleStride;
    const bool mine = (int)blockIdx.y < batch.n && kb < batch.layer[blockIdx.y].KB;
    // x may be the previous kernel's output: wait for it.  The main kernel that
    // follows prefetches weights as soon as this grid lets it launch, so unless
    // every kernel before is known never to write weights (early_trigger, inside
    // one decode stream) it is let launch only after that wait.
    if (batch.early_trigger) griddep_launch_dependents();
    griddep_wait();
    if (!batch.early_trigger) griddep_launch_dependents();
    if (mine) {
        const PrepLayer& L = batch.layer[blockIdx.y];
        prep_pair(L, kb, tok, lane, load_pair(L, kb, tok, lane));
    }
}

cudaError_t launch_linear_fp8(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                              const CUtensorMap& ts, const LinearParams& p, int grid, size_t smem,
                              cudaStream_t stream, bool launch) {
    return launch_family<kFP8>(family, mt, tw, tx, ts, p, grid, smem, stream, launch);
}

// One layer per launch passes a small parameter block (NB = 1); batches up to
// kMaxPrepLayers.
template <int NB>
static cudaError_t launch_prep_n(const PrepBatch& b, bool early_trigger, cudaStream_t stream) {
    // One warp per (k-block, token slot), 8 warps per block; one grid row per layer.
    PrepBatchN<NB> bb{};
    bb.n = b.n;
    bb.early_trigger = early_trigger ? 1 : 0;
    bb.wait_last = b.wait_last;
    int most = 1, total = 0;
    for (int i = 0; i < b.n; ++i) {
        bb.layer[i] = b.layer[i];
        bb.layer[i].pair0 = total;
        total += b.layer[i].KB * kUnscaleStride;
        const int blocks = (b.layer[i].KB * kUnscaleStride + 7) / 8;
        most = blocks > most ? blocks : most;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)most, (unsigned)b.n);
    if (b.wait_last) {
        int sms = 0, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int blocks = (total + 7) / 8;
        cfg.gridDim = dim3((unsigned)(blocks < sms ? blocks : sms), 1u);
    }
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, prep_x_kernel<NB>, bb);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_prep_x(const PrepBatch& b, bool early_trigger, cudaStream_t stream) {
    if (b.n < 1 || b.n > kMaxPrepLayers) return cudaErrorInvalidValue;
    // Copies made ahead (wait_last) run only in the batched instance, whatever
    // the number of layers: the single-layer instance has one warp per pair
    // and no grid-stride walk, so on the small grid it would leave pairs out.
    return (b.n == 1 && !b.wait_last) ? launch_prep_n<1>(b, early_trigger, stream)
                                      : launch_prep_n<kMaxPrepLayers>(b, early_trigger, stream);
}

}  // namespace dl
