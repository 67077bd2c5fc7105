// Internal interface between the C-ABI host code and the kernel translation
// units (not installed, not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dl {

struct LinearParams;

// Shared-memory bytes of one pipeline stage and the per-CTA fixed part, for a
// kernel staging `mt` token rows (mt in {1,2,4,8,16}).
int host_stage_bytes(int dtype, int mt);
int host_fixed_smem_bytes(int mt, int stages);
int host_x_rows(int mt);

// Launch the (dtype, family, mt) instance (launch = false: only raise its
// shared-memory ceiling on the current device, which is done once per device
// and never during stream capture).  Returns the first CUDA error.
cudaError_t launch_linear_bf16(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                               const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                               bool launch);
cudaError_t launch_linear_fp8(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                              const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                              bool launch);

}  // namespace dl
