// Launches of the tensor-core GEMM in CTA pairs (tcgen05 .cta_group::2, Q4_0
// weights): one translation unit of their own, so that they compile in
// parallel with the single-CTA instantiations.
#include "gemm_tc.cuh"

namespace pf {

cudaError_t launch_gemm_pair(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                             int withhold_stage, bool two) {
#define PF_PAIR_CASE(BNV)                                                              \
  if (W.BN == BNV)                                                                     \
    return two ? launch_t<W_Q4, BNV, 2, true>(A, M, W, ep, err, s, withhold_stage)    \
               : launch_t<W_Q4, BNV, 1, true>(A, M, W, ep, err, s, withhold_stage);
  PF_PAIR_CASE(128)
  PF_PAIR_CASE(192)
  PF_PAIR_CASE(256)
#undef PF_PAIR_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pf
