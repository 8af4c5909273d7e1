// w4_tc2.cu — the two-issuer variant of the tensor-core kernel (see
// w4_tc_kernel.cuh), compiled apart from the one-issuer kernels.
#include "w4_tc_kernel.cuh"

namespace w4 {

cudaError_t launch_tc_mma2(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                           const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s) {
  return launch_tc_t<true>(plan, amap, smap, zmap, args, s);
}

}  // namespace w4
