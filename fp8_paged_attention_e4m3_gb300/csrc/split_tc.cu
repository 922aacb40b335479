// Host launcher of the tcgen05 split kernel: builds the TMA tensor map of the
// KV pool and picks the instantiation for (head dim, padded rows).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "split_tc.cuh"

namespace vae4 {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

}  // namespace

unsigned long long current_context_id() {
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  });
  CUcontext c = nullptr;
  if (!g_ctx_current || !g_ctx_id || g_ctx_current(&c) != CUDA_SUCCESS || !c) return 0;
  unsigned long long id = 0;
  if (g_ctx_id(c, &id) != CUDA_SUCCESS) return 0;
  return id;
}

void tc_row_groups(int rows, int *n_rg, int *n) {
  const int g = (rows + 63) / 64;
  *n_rg = g;
  *n = ((rows + g - 1) / g + 15) / 16 * 16;
}

cudaError_t launch_split_tc(const SplitParams &p, long long wait_limit, cudaStream_t stream) {
  int n_rg = 1, n = 16;
  tc_row_groups(p.rows, &n_rg, &n);
  if (n_rg * n > p.rows_pad) return cudaErrorInvalidValue;  // workspace rows
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const int D = p.D;
  const int IB = D < 128 ? D : 128;
  TcArgs a;
  a.rows_total = p.n_pages * 2 * (int64_t)p.Hkv * p.page;
  a.wait_limit = wait_limit;
  a.drain_limit = 2000000000LL;  // about a second: copies and MMAs always finish
  a.n_rg = n_rg;
  if (a.rows_total > (int64_t)0x7fffff00) return cudaErrorInvalidValue;
  // the pool as a 3-D tensor: (byte within an IB-wide block, row of D bytes,
  // block of the row); a box of {IB, 16, D/IB} is one 16-key page slice
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)IB, (cuuint64_t)a.rows_total, (cuuint64_t)(D / IB)};
  const cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)IB};
  const cuuint32_t box[3] = {(cuuint32_t)IB, 16u, (cuuint32_t)(D / IB)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = encode(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                            const_cast<uint8_t *>(p.kv), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE,
                            IB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if (p.dev_plan) return launch_split_tc_dev(p, a, n, map, stream);
  if (p.t_from_len) return launch_split_tc_len(p, a, n, map, stream);
  return p.hilo ? launch_tc_any<kPlanFixed, true>(p, a, n, map, stream)
                : launch_tc_any<kPlanFixed, false>(p, a, n, map, stream);
}

}  // namespace vae4
