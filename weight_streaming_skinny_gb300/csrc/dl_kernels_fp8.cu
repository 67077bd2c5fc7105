// FP8 (e4m3, 128x128 block scales) instances of the decode-linear kernel.
#include "dl_kernels_common.cuh"

namespace dl {

cudaError_t launch_linear_fp8(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                              const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                              bool launch) {
    return launch_family<kFP8>(family, mt, tw, tx, p, grid, smem, stream, launch);
}

}  // namespace dl
