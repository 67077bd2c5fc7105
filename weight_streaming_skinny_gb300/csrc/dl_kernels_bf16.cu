// bf16-weight instances of the decode-linear kernel.
#include "dl_kernels_common.cuh"

namespace dl {

cudaError_t launch_linear_bf16(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                               const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                               bool launch) {
    return launch_family<kBF16>(family, mt, tw, tx, p, grid, smem, stream, launch);
}

int host_stage_bytes(int dtype, int mt) {
    const int xr = mt < 8 ? 8 : mt;
    return kBN * kBK * (dtype == kBF16 ? 2 : 1) + xr * kBK * 2;
}

int host_x_rows(int mt) { return mt < 8 ? 8 : mt; }

int host_fixed_smem_bytes(int mt, int stages) {
    return host_x_rows(mt) * kRedStride * 4 + stages * 16 + 16;
}

}  // namespace dl
