// Internal interface between the C-ABI host code and the kernel translation
// units (not installed, not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dl {

struct LinearParams;

// Dynamic shared memory of one CTA of the (dtype, family, mt) kernel with
// `stages` pipeline stages, and the token rows it stages (mt in {1,2,4,8,16}).
int host_smem_bytes(int dtype, int family, int mt, int stages);
int host_x_rows(int mt);
// CTAs per SM the (dtype, family, mt) kernel is compiled to fit.
int host_min_blocks(int dtype, int family, int mt);

// Launch the (dtype, family, mt) instance (launch = false: only raise its
// shared-memory ceiling on the current device, which is done once per device
// and never during stream capture).  Returns the first CUDA error.  tw: the
// weights, tx: the activations (FP8: their f16 copy or e4m3 parts), ts (FP8):
// the block scales as a one-dimensional fp32 map (boxes of 8).
cudaError_t launch_linear_bf16(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                               const LinearParams& p, int grid, size_t smem, cudaStream_t stream,
                               bool launch);
cudaError_t launch_linear_fp8(int family, int mt, const CUtensorMap& tw, const CUtensorMap& tx,
                              const CUtensorMap& ts, const LinearParams& p, int grid, size_t smem,
                              cudaStream_t stream, bool launch);

// FP8 activation prep of up to kMaxPrepLayers layers in one launch: for each,
// x (bf16 [M][K]) -> xh (f16 [KB][2][mtb][64], exact per-block power-of-two
// scaling, rows >= M zero; or, parts = 1, three e4m3 parts [KB][3][mtb][128]
// for the tensor-memory family) and unscale[KB][16]; K % 128 == 0.
constexpr int kMaxPrepLayers = 16;
struct PrepLayer {
    const uint16_t* x;
    uint16_t* xh;
    float* unscale;
    int M, K, KB, mtb;
    int pair0;                // set by launch_prep_x: first pair of this layer in the batch
    int parts;                // 0: the f16 copy; 1: the e4m3 parts
};
constexpr int kPrepInFlight = 8;
template <int NB>
struct PrepBatchN {
    PrepLayer layer[NB];
    int n;
    int early_trigger;
    // 1: every layer's x is known ready when the grid starts (no kernel still
    // running may write it): copy first, then wait for the previous kernel, so
    // the copy overlaps it while a kernel that waits for this grid still waits
    // for the previous one too.
    int wait_last;
};
using PrepBatch = PrepBatchN<kMaxPrepLayers>;
// early_trigger: let the next kernel launch before this one's wait (only when
// no kernel before it on the stream writes weights or scales).
cudaError_t launch_prep_x(const PrepBatch& b, bool early_trigger, cudaStream_t stream);

}  // namespace dl
