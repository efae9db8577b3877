// Launches of the tensor-core GEMM whose CTAs take one work unit each (Q4_0
// weights): the epilogue stages in the dequantised-B ring and the A ring
// gets one more stage.  A translation unit of their own, so that they
// compile in parallel with the other instantiations.
#include "gemm_tc.cuh"

namespace pf {

template <int BN, int MT>
static bool fits(int split) {
  using C = GemmCfg<W_Q4, BN, MT, false, true>;
  return static_cast<size_t>(split - 1) * 128 * BN * 4 <= static_cast<size_t>(C::S_A) * C::A_STAGE;
}

bool gemm_solo_fits(int BN, bool two, int split) {
  switch (BN) {
    case 64: return two ? fits<64, 2>(split) : fits<64, 1>(split);
    case 128: return two ? fits<128, 2>(split) : fits<128, 1>(split);
    case 192: return two ? fits<192, 2>(split) : fits<192, 1>(split);
    case 256: return two ? fits<256, 2>(split) : fits<256, 1>(split);
    default: return false;
  }
}

cudaError_t launch_gemm_solo(const ActMat& A, int M, const WeightMat& W, const EpiParams& ep, int* err, cudaStream_t s,
                             int withhold_stage, bool two) {
#define PF_SOLO_CASE(BNV)                                                                \
  if (W.BN == BNV)                                                                       \
    return two ? launch_t<W_Q4, BNV, 2, false, true>(A, M, W, ep, err, s, withhold_stage) \
               : launch_t<W_Q4, BNV, 1, false, true>(A, M, W, ep, err, s, withhold_stage);
  PF_SOLO_CASE(64)
  PF_SOLO_CASE(128)
  PF_SOLO_CASE(192)
  PF_SOLO_CASE(256)
#undef PF_SOLO_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pf
