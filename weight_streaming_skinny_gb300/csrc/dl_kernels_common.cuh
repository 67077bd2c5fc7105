// Instantiation helper shared by the per-dtype kernel translation units.
#pragma once

#include <atomic>

#include "dl_kernel.cuh"
#include "dl_launch.h"

namespace dl {

// Raise the instance's dynamic shared-memory ceiling to `smem` on the current
// device, once per device (a host-side function attribute, never enqueued).
template <int DT, int FAM, int MT>
cudaError_t prepare_instance(size_t smem) {
    static std::atomic<int> set_bytes[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (set_bytes[dev].load() >= (int)smem) return cudaSuccess;
    e = cudaFuncSetAttribute(linear_kernel<DT, FAM, MT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) set_bytes[dev].store((int)smem);
    return e;
}

template <int DT, int FAM, int MT>
cudaError_t launch_instance(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts,
                            const LinearParams& p,
                            int grid, size_t smem, cudaStream_t stream, bool launch) {
    cudaError_t e = prepare_instance<DT, FAM, MT>(smem);
    if (e != cudaSuccess || !launch) return e;
    // Programmatic stream serialization: this grid may start while the
    // previous kernel on the stream drains; the kernel orders every dependent
    // access after griddepcontrol.wait.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads_for(DT, FAM));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, linear_kernel<DT, FAM, MT>, tw, tx, ts, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_family(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                          const CUtensorMap& ts,
                          const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                          bool launch) {
    if (family == kMMA) {
        if (mt == 8) return launch_instance<DT, kMMA, 8>(tw, tx, ts, p, grid, smem, stream, launch);
        if (mt == 16) return launch_instance<DT, kMMA, 16>(tw, tx, ts, p, grid, smem, stream, launch);
        return cudaErrorInvalidValue;
    }
    if (family == kTC) {
        // tensor-memory family: FP8 weights only (kind::f8f6f4 MMAs)
        if constexpr (DT == kFP8) {
            if (mt == 8) return launch_instance<DT, kTC, 8>(tw, tx, ts, p, grid, smem, stream, launch);
            if (mt == 16) return launch_instance<DT, kTC, 16>(tw, tx, ts, p, grid, smem, stream, launch);
        }
        return cudaErrorInvalidValue;
    }
    switch (mt) {
        case 1: return launch_instance<DT, kSIMT, 1>(tw, tx, ts, p, grid, smem, stream, launch);
        case 2: return launch_instance<DT, kSIMT, 2>(tw, tx, ts, p, grid, smem, stream, launch);
        default: break;
    }
    if constexpr (DT == kBF16) {
        // FP8 SIMT stops at 2 tokens (the host plan switches to MMA beyond).
        if (mt == 4) return launch_instance<DT, kSIMT, 4>(tw, tx, ts, p, grid, smem, stream, launch);
        if (mt == 8) return launch_instance<DT, kSIMT, 8>(tw, tx, ts, p, grid, smem, stream, launch);
        if (mt == 16) return launch_instance<DT, kSIMT, 16>(tw, tx, ts, p, grid, smem, stream, launch);
    }
    return cudaErrorInvalidValue;
}

}  // namespace dl
