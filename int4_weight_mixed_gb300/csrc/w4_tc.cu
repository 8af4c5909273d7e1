// w4_tc.cu — the tensor-core schedule of the 4-bit-weight GEMM for sm_103a:
// shared-memory sizing, the one-issuer kernel instantiations and the launch
// dispatch (the kernel itself is in w4_tc_kernel.cuh; the two-issuer variant
// is compiled in w4_tc2.cu, the CTA-pair variant in w4_tc3.cu).
#include "w4_tc_kernel.cuh"

namespace w4 {

// wblk: prepacked weight bytes of one K block of one 128-column tile (4096
// for 64-K blocks, 8192 for the 128-K blocks of fp8 activations)
size_t tc_stage_bytes(int bm, int nsub, int nt, int wblk) {
  return static_cast<size_t>(nsub) *
         (static_cast<size_t>(bm) * 128 + static_cast<size_t>(nt) * (wblk + 256 + 256));
}

size_t tc_smem_bytes(int bm, int nsub, int nt, int stages, int wblk) {
  const size_t bars = (2 * kMaxStages + kMaxTmemStages + 3) * 8;
  return 1024 + tc_stage_bytes(bm, nsub, nt, wblk) * stages + bars + 64;  // + slot, abort, tok[2]
}

// Most pipeline stages that fit in shared memory (0 when none does).
int tc_max_stages(int bm, int nsub, int nt, int wblk) {
  const size_t budget = 225 * 1024;
  int s = kMaxStages;
  while (s > 0 && tc_smem_bytes(bm, nsub, nt, s, wblk) > budget) --s;
  return s;
}

cudaError_t launch_tc_mma2(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                           const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s);
cudaError_t launch_tc_pair(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                           const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s);

cudaError_t launch_tc(const TcPlan& plan, const CUtensorMap& amap, const CUtensorMap& smap,
                      const CUtensorMap& zmap, const TcArgs& args, cudaStream_t s) {
  if (plan.pair) return launch_tc_pair(plan, amap, smap, zmap, args, s);
  if (!tc_mma2(plan)) return launch_tc_t<false>(plan, amap, smap, zmap, args, s);
  return launch_tc_mma2(plan, amap, smap, zmap, args, s);
}

}  // namespace w4
