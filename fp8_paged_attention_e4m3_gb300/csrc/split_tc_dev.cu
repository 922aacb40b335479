// The tcgen05 split kernel's device-side-plan instantiations, in a
// translation unit of their own so the plan modes compile in parallel.
#include "split_tc.cuh"

namespace vae4 {

cudaError_t launch_split_tc_dev(const SplitParams &p, const TcArgs &a, int n,
                                const CUtensorMap &map_k, const CUtensorMap &map_v,
                                cudaStream_t stream) {
  return p.hilo ? launch_tc_any<kPlanDevice, true>(p, a, n, map_k, map_v, stream)
                : launch_tc_any<kPlanDevice, false>(p, a, n, map_k, map_v, stream);
}

}  // namespace vae4
