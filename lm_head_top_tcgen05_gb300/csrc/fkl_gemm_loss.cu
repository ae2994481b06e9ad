// Instantiations of the persistent tcgen05 GEMM with the loss epilogues: the forward
// projection + online logsumexp + top-K gather, and the backward recompute + dS.
#include "fkl_gemm.cuh"

namespace fkl {

cudaError_t launch_gemm_fwd(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                            const FwdParams& ep, int grid, cudaStream_t st) {
  return launch_gemm_t<kVocabTile, false, false, EpiFwd>(a, b, g, ep, grid, st);
}

cudaError_t launch_gemm_ds(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                           const DsParams& ep, int grid, cudaStream_t st) {
  return launch_gemm_t<kVocabTile, false, false, EpiDs>(a, b, g, ep, grid, st);
}

}  // namespace fkl
