// fkl_forward_noalloc: the forward pass for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a workspace: a plugin or custom operator living inside
// another runtime that owns the whole device memory pool and hands out only the tensors of
// the op's inputs and outputs, or a latency-critical loop that must never call cudaMalloc
// (which can synchronise the device and can fail once the pool is carved up).  For them
// this file keeps the forward's scratch in a fixed, file-scope device array that the CUDA
// runtime reserves when the library's module is loaded on a device.  Every GPU that loads
// the library keeps this array until the process exits.
//
// The array's name is only a host-side stand-in for the device symbol: host code must not
// hand it to a kernel.  Its device address is looked up with cudaGetSymbolAddress, with the
// device current.  The first call on a device does the set-up (the library's module is
// loaded there, and the device's compute capability and SM count are read and kept); every
// call repeats the address lookup, which is cheap once the module is loaded and allocates
// nothing, so that a context re-created after cudaDeviceReset never sees a stale address.
#include <cstdio>
#include <mutex>

#include "../../include/fkl.h"
#include "fkl_internal.h"

namespace fkl {

// Largest forward scratch the static array holds: 64 MiB.  The forward needs about
// T * (8K + 400) bytes (sorted teacher pairs, entropy terms, token weights and counts,
// per-split partials, block sums), so T up to about 56K tokens at K = 100.
constexpr size_t kNoAllocScratchBytes = size_t{64} << 20;

static __device__ __align__(256) unsigned char fkl_static_scratch[kNoAllocScratchBytes];

static fkl_status noalloc_fail(fkl_status s, const char* msg) {
  set_last_error_message(msg);
  return s;
}

// Device address of the static scratch on the current device.  The device check and SM count
// are taken once per device; the address is looked up on every call.
static fkl_status scratch_address(uint8_t** out, int* sms) {
  static std::mutex mu;
  static int sm_count[128] = {};  // 0: this device not set up yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128)
    return noalloc_fail(FKL_ERR_CUDA, "cudaGetDevice failed");
  {
    std::lock_guard<std::mutex> lk(mu);
    if (sm_count[dev] == 0) {
      int major = 0, minor = 0, n = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return noalloc_fail(FKL_ERR_CUDA, "cudaDeviceGetAttribute failed");
      if (major != 10 || minor != 3) return noalloc_fail(FKL_ERR_UNSUPPORTED, "device is not sm_103");
      sm_count[dev] = n;
    }
    *sms = sm_count[dev];
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, fkl_static_scratch);
  if (e != cudaSuccess || p == nullptr)
    return noalloc_fail(FKL_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
  *out = static_cast<uint8_t*>(p);
  return FKL_OK;
}

}  // namespace fkl

using namespace fkl;

extern "C" fkl_status fkl_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                                          const float* topk_logits, const uint8_t* mask, int64_t T,
                                          int64_t d, int64_t V, int64_t K, float tau, float* loss,
                                          float* lse, void* stream) {
  set_last_error_message("");
  Plan pl;
  // the one-SM forward deals its units round-robin: at most kMaxDealtSplit partials per row
  if (!make_plan(T, d, V, K, 1, &pl, false, kMaxDealtSplit)) return noalloc_fail(FKL_ERR_INVALID_ARG, "unsupported shape");
  if (!(tau > 0.f) || tau == INFINITY) return noalloc_fail(FKL_ERR_INVALID_ARG, "tau must be finite and > 0");
  if (W == nullptr || loss == nullptr || (T > 0 && (H == nullptr || topk_idx == nullptr || topk_logits == nullptr || lse == nullptr)))
    return noalloc_fail(FKL_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(H) | reinterpret_cast<uintptr_t>(W)) % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(topk_idx) | reinterpret_cast<uintptr_t>(topk_logits) |
       reinterpret_cast<uintptr_t>(loss) | reinterpret_cast<uintptr_t>(lse)) % 4 != 0)
    return noalloc_fail(FKL_ERR_ALIGNMENT, "H and W need 16-byte alignment, the rest 4-byte");
  // The forward uses the workspace up to the backward-only dS slab.
  const size_t need = pl.off_ds;
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "this shape needs %zu bytes of forward scratch; the static scratch holds %zu bytes "
             "(about T * (8K + 400) bytes are needed)", need, kNoAllocScratchBytes);
    return noalloc_fail(FKL_ERR_WORKSPACE, msg);
  }
  uint8_t* ws = nullptr;
  int sms = 0;
  fkl_status s = scratch_address(&ws, &sms);
  if (s != FKL_OK) return s;
  {
    const NamedPtr ptrs[] = {{H, "H"}, {W, "W"}, {topk_idx, "topk_idx"}, {topk_logits, "topk_logits"},
                             {mask, "mask"}, {loss, "loss"}, {lse, "lse"}};
    if ((s = static_cast<fkl_status>(check_device_memory(ptrs))) != FKL_OK) return s;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  // The header (status word) must start at zero; every other region is fully rewritten.
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return noalloc_fail(FKL_ERR_CUDA, "cudaMemsetAsync failed");
  int2* pairs = reinterpret_cast<int2*>(ws + pl.off_pairs);
  float* crow = reinterpret_cast<float*>(ws + pl.off_crow);
  float* part = reinterpret_cast<float*>(ws + pl.off_part);
  double* bsum = reinterpret_cast<double*>(ws + pl.off_bsum);
  int* bcnt = reinterpret_cast<int*>(ws + pl.off_bcnt);
  float* wrow = reinterpret_cast<float*>(ws + pl.off_wrow);
  if (T == 0) {
    if (launch_combine(part, 1, crow, wrow, 0, tau, lse, bsum, bcnt, 0, hdr, loss, st) != cudaSuccess)
      return noalloc_fail(FKL_ERR_CUDA, "combine launch failed");
    return FKL_OK;
  }
  if (launch_prep(topk_idx, topk_logits, T, (int)K, (int)V, tau, pairs, nullptr, crow, &hdr->status, st) != cudaSuccess)
    return noalloc_fail(FKL_ERR_CUDA, "prep launch failed");
  if (launch_weights(mask, nullptr, 1, 0, T, reinterpret_cast<int*>(ws + pl.off_scnt), hdr, wrow, nullptr, st) !=
      cudaSuccess)
    return noalloc_fail(FKL_ERR_CUDA, "weights launch failed");
  CUtensorMap mH, mW;
  if (!encode_map_bf16(&mH, H, d, T, d * 2, 64, 128) || !encode_map_bf16(&mW, W, d, V, d * 2, 64, kVocabTile))
    return noalloc_fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  const int m_tiles = static_cast<int>((T + 127) / 128);
  const int n_tiles = static_cast<int>((V + kVocabTile - 1) / kVocabTile);
  const int nsplit = plan_splits(m_tiles, n_tiles, sms);
  const GemmShape g = make_shape(T, V, d, kVocabTile, nsplit, &hdr->status);
  FwdParams fp;
  fp.pairs = pairs;
  fp.part = part;
  fp.sg = nullptr;
  fp.T = (int)T; fp.K = (int)K; fp.V = (int)V; fp.nsplit = nsplit;
  fp.scale2 = kLog2e / tau;
  if (launch_gemm_fwd(mH, mW, g, fp, g.num_units < sms ? g.num_units : sms, st) != cudaSuccess)
    return noalloc_fail(FKL_ERR_CUDA, "forward GEMM launch failed");
  if (launch_combine(part, nsplit, crow, wrow, T, tau, lse, bsum, bcnt, pl.nb, hdr, loss, st) != cudaSuccess)
    return noalloc_fail(FKL_ERR_CUDA, "combine launch failed");
  return FKL_OK;
}
