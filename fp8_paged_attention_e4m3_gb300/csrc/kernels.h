// Launchers of the library's kernels (internal; the public ABI is in
// include/verify_attn_e4m3.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "params.h"

namespace vae4 {

// Split kernel on the warp-level (mma.sync) tensor-core path.
size_t split_mma_smem_bytes(int D, int rows_pad);
int split_mma_threads(int rows_pad);
cudaError_t launch_split_mma(const SplitParams &p, cudaStream_t stream);

// Combine kernel (programmatic dependent launch after the split kernel).
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);

// Decode-table test hook.
cudaError_t launch_decode_table(uint16_t *out, cudaStream_t stream);

}  // namespace vae4
