// bf16-weight instances of the decode-linear kernel.
#include "dl_kernels_common.cuh"

namespace dl {

cudaError_t launch_linear_bf16(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                               const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                               bool launch) {
    // (bf16 has no block scales: the kernel never reads its third map)
    return launch_family<kBF16>(family, mt, tw, tx, tx, p, grid, smem, stream, launch);
}

int host_smem_bytes(int dtype, int family, int mt, int stages) {
    return smem_layout(dtype, family, mt, stages).total + 1024;   // + alignment slack
}

int host_x_rows(int mt) { return mt < 8 ? 8 : mt; }

int host_min_blocks(int dtype, int family, int mt) { return min_blocks_for(dtype, family, mt); }

}  // namespace dl
