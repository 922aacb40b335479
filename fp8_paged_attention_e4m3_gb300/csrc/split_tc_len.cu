// The tcgen05 split kernel's instantiations for a static grid whose
// partition length follows each sequence's length (the automatic plan of a
// single sequence), in a translation unit of their own so the plan modes
// compile in parallel.
#include "split_tc.cuh"

namespace vae4 {

cudaError_t launch_split_tc_len(const SplitParams &p, const TcArgs &a, int n,
                                const CUtensorMap &map_k, const CUtensorMap &map_v,
                                cudaStream_t stream) {
  return p.hilo ? launch_tc_any<kPlanFromLen, true>(p, a, n, map_k, map_v, stream)
                : launch_tc_any<kPlanFromLen, false>(p, a, n, map_k, map_v, stream);
}

}  // namespace vae4
