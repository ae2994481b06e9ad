// Instantiations of the two-SM (cta_group::2) persistent GEMM: the loss's forward and dS
// epilogues with 256 x 256 tiles, and the fp32 epilogue for dW / dH and the test hook; and
// the fixup that completes K-split fp32 units.
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
  if (ep.out16 != nullptr) {  // bf16 destination: the backward's dW (A, B MN-major) and dH (B MN-major)
    if (a_mn && b_mn) return launch_gemm2_t<BN, true, true, EpiF32Bf16>(a, b, g, ep, sms, st);
    if (!a_mn && b_mn) return launch_gemm2_t<BN, false, true, EpiF32Bf16>(a, b, g, ep, sms, st);
    return cudaErrorInvalidValue;
  }
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

// One block per (split unit, slice of its rows): sums the unit's K pieces in piece order and
// stores, or adds, the tile into the product's output.  BN columns per tile.
__global__ void __launch_bounds__(256) ksplit_fixup_kernel(const GemmShape g, const F32Params p, int bn) {
  const int r = static_cast<int>(blockIdx.x);
  int m_blk, nb, ne, split;
  unit_range(g, g.split_from + r, m_blk, nb, ne, split);
  const size_t tile = static_cast<size_t>(kBM2) * bn;
  const float* part = g.kpart + static_cast<size_t>(r) * g.ksplit * tile;
  const int cols4 = bn / 4;
  const int total = kBM2 * cols4;
  for (int i = static_cast<int>(blockIdx.y * blockDim.x + threadIdx.x); i < total;
       i += static_cast<int>(gridDim.y * blockDim.x)) {
    const int tr = i / cols4;
    const int tc = (i - tr * cols4) * 4;
    const int row = m_blk * kBM2 + tr;
    const int col = nb * bn + tc;
    if (row >= p.M || col >= p.N) continue;
    const float* src = part + static_cast<size_t>(tr) * bn + tc;
    float4 s = *reinterpret_cast<const float4*>(src);
    for (int q = 1; q < g.ksplit; ++q) {
      const float4 y = *reinterpret_cast<const float4*>(src + q * tile);
      s.x += y.x; s.y += y.y; s.z += y.z; s.w += y.w;
    }
    if (p.out16 != nullptr) {  // bf16 destination: (fp32 sum so far +) pieces, rounded once
      float sv[4] = {s.x, s.y, s.z, s.w};
      const float* src = p.accumulate ? p.out + static_cast<size_t>(row) * p.ldo + col : nullptr;
      uint16_t* o16 = p.out16 + static_cast<size_t>(row) * p.ldo16 + col;
      for (int j = 0; j < 4 && col + j < p.N; ++j) {
        const float x = src != nullptr ? src[j] + sv[j] : sv[j];
        o16[j] = static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
      }
      continue;
    }
    float* o = p.out + static_cast<size_t>(row) * p.ldo + col;
    if (p.vec_ok && col + 4 <= p.N) {
      float4* o4 = reinterpret_cast<float4*>(o);
      if (p.accumulate) {
        const float4 y = *o4;
        s.x += y.x; s.y += y.y; s.z += y.z; s.w += y.w;
      }
      *o4 = s;
    } else {
      const float sv[4] = {s.x, s.y, s.z, s.w};
      for (int j = 0; j < 4 && col + j < p.N; ++j) o[j] = p.accumulate ? o[j] + sv[j] : sv[j];
    }
  }
}

cudaError_t launch_ksplit_fixup(int bn, const GemmShape& g, const F32Params& ep, cudaStream_t st) {
  const int units = g.num_units - g.split_from;
  if (units <= 0 || g.ksplit < 2) return cudaSuccess;
  ksplit_fixup_kernel<<<dim3(static_cast<unsigned>(units), 16), 256, 0, st>>>(g, ep, bn);
  return cudaGetLastError();
}

}  // namespace fkl
