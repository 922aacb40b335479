// Launchers of the library's kernels (internal; the public ABI is in
// include/verify_attn_e4m3.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "params.h"

namespace vae4 {

// Unique id of the CUDA context current on the calling thread (0 if none
// is current or the driver cannot tell).  Per-device caches of the host
// code (function attributes, symbol addresses) are keyed on it, so that a
// context created after cudaDeviceReset is set up afresh.
unsigned long long current_context_id();

// Split kernel on the warp-level (mma.sync) tensor-core path.
size_t split_mma_smem_bytes(int D, int rows_pad);
int split_mma_threads(int rows_pad);
cudaError_t launch_split_mma(const SplitParams &p, cudaStream_t stream);

// Split kernel on the tcgen05 tensor cores (TMA + TMEM); the default path.
// wait_limit: SM cycles after which a pipeline wait gives up.
cudaError_t launch_split_tc(const SplitParams &p, long long wait_limit, cudaStream_t stream);
// Row groups of the tcgen05 kernel: rows are processed in n_rg groups of n
// (a multiple of 16, at most 64) rows; the workspace needs n_rg * n rows.
void tc_row_groups(int rows, int *n_rg, int *n);

// Combine kernel (programmatic dependent launch after the split kernel).
cudaError_t launch_combine(const CombineParams &p, cudaStream_t stream);
cudaError_t launch_kv_read(const SplitParams &p, int num_sms, cudaStream_t stream);
cudaError_t launch_bridge(const BridgeParams &p, int num_sms, bool e5m2, bool raw,
                          cudaStream_t stream);

// Decode-table test hook.
cudaError_t launch_decode_table(uint16_t *out, bool integer_path, bool e5m2,
                                cudaStream_t stream);

}  // namespace vae4
