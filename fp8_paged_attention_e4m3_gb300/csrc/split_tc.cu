// Host launcher of the tcgen05 split kernel: builds the TMA tensor map of the
// KV pool and picks the instantiation for (head dim, padded rows).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include <string.h>

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

// The 5-D tensor map of one cache (K or V): coordinates (byte within an
// IB-wide block, token in the page, block of the key row, KV head, page),
// strides (token, IB, head, page) in bytes; a box {IB, 16, D/IB, 1, 1} is
// one 16-key slice of one head, laid out in shared memory as D/IB blocks of
// 16 rows x IB bytes (swizzled) whatever the cache's layout.
bool encode_cache_map(CUtensorMap *map, const uint8_t *base, int64_t ps, int64_t ts, int64_t hs,
                      const SplitParams &p) {
  auto encode = encode_fn();
  if (!encode) return false;
  const int D = p.D, IB = D < 128 ? D : 128;
  const cuuint64_t dims[5] = {(cuuint64_t)IB, (cuuint64_t)p.page, (cuuint64_t)(D / IB),
                              (cuuint64_t)p.Hkv, (cuuint64_t)p.n_pages};
  const cuuint64_t strides[4] = {(cuuint64_t)ts, (cuuint64_t)IB, (cuuint64_t)hs, (cuuint64_t)ps};
  const cuuint32_t box[5] = {(cuuint32_t)IB, 16u, (cuuint32_t)(D / IB), 1u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<uint8_t *>(base), dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                IB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_describable(const uint8_t *base, int64_t ps, int64_t ts, int64_t hs) {
  return (reinterpret_cast<uintptr_t>(base) & 15u) == 0 && ps % 16 == 0 && ts % 16 == 0 &&
         hs % 16 == 0 && ps < ((int64_t)1 << 40) && ts < ((int64_t)1 << 40) &&
         hs < ((int64_t)1 << 40);
}

cudaError_t launch_split_tc(const SplitParams &p_in, long long wait_limit, cudaStream_t stream) {
  int n_rg = 1, n = 16;
  tc_row_groups(p_in.rows, &n_rg, &n);
  if (n_rg * n > p_in.rows_pad) return cudaErrorInvalidValue;  // workspace rows
  if (p_in.n_pages > 0x7fffffff) return cudaErrorInvalidValue;  // 32-bit page coordinate
  SplitParams p = p_in;
  TcArgs a;
  a.wait_limit = wait_limit;
  a.drain_limit = 2000000000LL;  // about a second: copies and MMAs always finish
  a.n_rg = n_rg;
  // tensor loads when both caches can be described by tensor maps (16-byte
  // aligned base and strides), else 8-byte asynchronous copies
  CUtensorMap map_k, map_v;
  memset(&map_k, 0, sizeof(map_k));
  memset(&map_v, 0, sizeof(map_v));
  p.kv_cpasync = 1;
  if (tma_describable(p.k_base, p.k_ps, p.k_ts, p.k_hs) &&
      tma_describable(p.v_base, p.v_ps, p.v_ts, p.v_hs) &&
      encode_cache_map(&map_k, p.k_base, p.k_ps, p.k_ts, p.k_hs, p) &&
      encode_cache_map(&map_v, p.v_base, p.v_ps, p.v_ts, p.v_hs, p))
    p.kv_cpasync = 0;
  if (p.dev_plan) return launch_split_tc_dev(p, a, n, map_k, map_v, stream);
  if (p.t_from_len) return launch_split_tc_len(p, a, n, map_k, map_v, stream);
  return p.hilo ? launch_tc_any<kPlanFixed, true>(p, a, n, map_k, map_v, stream)
                : launch_tc_any<kPlanFixed, false>(p, a, n, map_k, map_v, stream);
}

}  // namespace vae4
