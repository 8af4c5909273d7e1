// w4_tc3.cu — the CTA-pair variant of the tensor-core kernel (two CTAs of a
// cluster share each tcgen05.mma, cta_group::2; see w4_tc_kernel.cuh),
// compiled apart from the other variants.
#include "w4_tc_kernel.cuh"

#ifndef W4_PAIR_MMA2
#define W4_PAIR_MMA2 1  // two alternating MMA issuers in rank 0
#endif

namespace w4 {

cudaError_t launch_tc_pair(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                           const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s) {
  // one 128-column weight tile per CTA of a pair (the kernel's tile geometry,
  // a compile-time constant in its LEAN instances)
  if (plan.nt != 1) return cudaErrorInvalidValue;
  if (W4_PAIR_MMA2) return launch_tc_t<true, true>(plan, amap, smap, zmap, args, s);
  return launch_tc_t<false, true>(plan, amap, smap, zmap, args, s);
}

int tc_pair_clusters(int mode, size_t smem) {
  switch (mode) {
    case kW4A16_F16: return tc_pair_clusters_mode<kW4A16_F16>(smem);
    case kW4A16_BF16: return tc_pair_clusters_mode<kW4A16_BF16>(smem);
    case kW4A8F8: return tc_pair_clusters_mode<kW4A8F8>(smem);
    default: return tc_pair_clusters_mode<kW4A8>(smem);
  }
}

}  // namespace w4
