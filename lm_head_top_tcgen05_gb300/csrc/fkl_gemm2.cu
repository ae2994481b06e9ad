// Instantiations of the two-SM (cta_group::2) persistent GEMM: the loss's forward and dS
// epilogues with 256 x 256 tiles, and the fp32 epilogue for dW / dH and the test hook.
#include "fkl_gemm2.cuh"

namespace fkl {

cudaError_t launch_gemm2_fwd(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                             const FwdParams& ep, int sms, cudaStream_t st) {
  return launch_gemm2_t<kVocabTile, false, false, EpiFwd>(a, b, g, ep, sms, st);
}

cudaError_t launch_gemm2_ds(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                            const DsParams& ep, int sms, cudaStream_t st) {
  return launch_gemm2_t<kVocabTile, false, false, EpiDs>(a, b, g, ep, sms, st);
}

template <int BN>
static cudaError_t dispatch2(bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmShape& g, const F32Params& ep, int sms, cudaStream_t st) {
  if (!a_mn && !b_mn) return launch_gemm2_t<BN, false, false, EpiF32>(a, b, g, ep, sms, st);
  if (!a_mn && b_mn) return launch_gemm2_t<BN, false, true, EpiF32>(a, b, g, ep, sms, st);
  if (a_mn && !b_mn) return launch_gemm2_t<BN, true, false, EpiF32>(a, b, g, ep, sms, st);
  return launch_gemm2_t<BN, true, true, EpiF32>(a, b, g, ep, sms, st);
}

cudaError_t launch_gemm2_f32(int bn, bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmShape& g, const F32Params& ep, int sms, cudaStream_t st) {
  switch (bn) {
    case 256: return dispatch2<256>(a_mn, b_mn, a, b, g, ep, sms, st);
    case 192: return dispatch2<192>(a_mn, b_mn, a, b, g, ep, sms, st);
    case 128: return dispatch2<128>(a_mn, b_mn, a, b, g, ep, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fkl
