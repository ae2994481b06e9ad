// One-SM instantiation of the forward projection + online logsumexp + top-K gather, used by
// the allocation-free forward (the loss itself runs on the two-SM kernel, fkl_gemm2.cu).
#include "fkl_gemm.cuh"

namespace fkl {

cudaError_t launch_gemm_fwd(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                            const FwdParams& ep, int grid, cudaStream_t st) {
  return launch_gemm_t<kVocabTile, false, false, EpiFwd>(a, b, g, ep, grid, st);
}

}  // namespace fkl
