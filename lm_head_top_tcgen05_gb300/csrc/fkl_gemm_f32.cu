// Instantiations of the persistent tcgen05 GEMM with a plain fp32 store/accumulate
// epilogue: the backward's dW = dS^T H (A and B MN-major) and dH += dS W (B MN-major),
// and every other major-ness / tile-width combination for the GEMM test hook.
#include "fkl_gemm.cuh"

namespace fkl {

template <int BN>
static cudaError_t dispatch_major(bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                                  const GemmShape& g, const F32Params& ep, int grid, cudaStream_t st) {
  if (!a_mn && !b_mn) return launch_gemm_t<BN, false, false, EpiF32>(a, b, g, ep, grid, st);
  if (!a_mn && b_mn) return launch_gemm_t<BN, false, true, EpiF32>(a, b, g, ep, grid, st);
  if (a_mn && !b_mn) return launch_gemm_t<BN, true, false, EpiF32>(a, b, g, ep, grid, st);
  return launch_gemm_t<BN, true, true, EpiF32>(a, b, g, ep, grid, st);
}

cudaError_t launch_gemm_f32(int bn, bool a_mn, bool b_mn, const CUtensorMap& a,
                            const CUtensorMap& b, const GemmShape& g, const F32Params& ep,
                            int grid, cudaStream_t st) {
  switch (bn) {
    case 256: return dispatch_major<256>(a_mn, b_mn, a, b, g, ep, grid, st);
    case 192: return dispatch_major<192>(a_mn, b_mn, a, b, g, ep, grid, st);
    case 128: return dispatch_major<128>(a_mn, b_mn, a, b, g, ep, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fkl
