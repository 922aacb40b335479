// Host launcher of the tcgen05 split kernel: builds the TMA tensor map of the
// KV pool and picks the instantiation for (head dim, padded rows).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
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

template <int D, int N>
cudaError_t launch(const SplitParams &p, const TcArgs &a, const CUtensorMap &map,
                   cudaStream_t stream) {
  using C = TcCfg<D, N>;
  // the shared-memory opt-in is a per-device function attribute: set it once
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(split_tc_kernel<D, N>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // programmatic dependent launch: the CTAs may be placed while the previous
  // kernel on the stream drains; the kernel waits for it before its first
  // global-memory access
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.P, p.Hkv * a.n_rg, p.B);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_tc_kernel<D, N>, p, a, map);
}

template <int D>
cudaError_t launch_d(const SplitParams &p, const TcArgs &a, int n, const CUtensorMap &map,
                     cudaStream_t stream) {
  switch (n) {
    case 16: return launch<D, 16>(p, a, map, stream);
    case 32: return launch<D, 32>(p, a, map, stream);
    case 48: return launch<D, 48>(p, a, map, stream);
    case 64: return launch<D, 64>(p, a, map, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

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
  switch (D) {
    case 64: return launch_d<64>(p, a, n, map, stream);
    case 128: return launch_d<128>(p, a, n, map, stream);
    case 256: return launch_d<256>(p, a, n, map, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace vae4
