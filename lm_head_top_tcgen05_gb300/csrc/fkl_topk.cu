// Offline teacher cache: the K largest teacher logits per position (fkl_teacher_topk).
//
// "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL
// Loss", section "Two systems changes", paragraph "Offline distillation": the teacher runs
// once and its top-100 tokens and logits per position are stored and reused.  Here the
// teacher's LM-head projection s = Ht Wt^T is fused with the selection, so the T x V logits
// are never written; two passes over the projection run on the two-SM GEMM:
//
//   1. bound pass   over every s-th vocabulary row of Wt (a strided tensor-map view; s
//                   up to kMaxBoundStride, as long as enough values are kept), each row
//                   keeps, per vocabulary split, its kTopR largest logits in registers
//                   (EpiTopR).  bound_kernel takes the K-th largest of those S * kTopR
//                   values: theta_t, a lower bound of the row's K-th largest logit (it is
//                   the K-th largest of a subset of the row).  About s * K logits of a row
//                   reach it, so the pass costs 1/s of a projection and the candidate
//                   buffer holds 4 s K.
//   2. candidate    recompute; every logit >= theta_t is appended to the row's candidate
//      pass         buffer (EpiCand; an integer atomic counter per row).  All of the row's
//                   top K are among them.
//   3. select       per row, rank the candidates by (logit descending, id ascending) and
//                   write the first K.  The ranks do not depend on the order of the appends,
//                   so the output is deterministic.
//
// A row with more candidates than the buffer holds (massive ties) is reported as
// FKL_ERR_TOPK_OVERFLOW and its outputs are set to id -1 and logit NaN.  For small
// vocabularies (V <= kAllCandidatesV) the bound pass is skipped and every logit of a row
// is a candidate.
#include <climits>
#include <cmath>
#include <mutex>

#include "../../include/fkl.h"
#include "fkl_gemm2.cuh"

namespace fkl {

constexpr int kTopR = 8;                // logits kept per (row, split) in the bound pass
constexpr int kMaxBoundSplits = 32;     // splits of the bound pass
constexpr int kMaxBoundStride = 8;      // the bound pass reads every s-th vocabulary row, s <= 8
constexpr int64_t kAllCandidatesV = 4096;

struct TopRParams {
  float* topr;  // [split][T][kTopR]
  int T, V;
};

struct CandParams {
  const float* theta;  // [T]
  int* cnt;            // [T]
  int2* cand;          // [T][cap]: (logit bits, id)
  int cap, T, V;
};

// ---------------------------------------------------------------- bound pass epilogue
struct EpiTopR {
  using Params = TopRParams;
  const Params& p;
  int t;
  bool row_ok;
  float r[kTopR];  // descending

  __device__ explicit EpiTopR(const Params& prm) : p(prm) {}

  __device__ __forceinline__ void begin_unit(int row0, int, int, int row) {
    t = row0 + row;
    row_ok = t < p.T;
#pragma unroll
    for (int i = 0; i < kTopR; ++i) r[i] = -INFINITY;
  }

  __device__ __forceinline__ void insert(float x) {
#pragma unroll
    for (int i = kTopR - 1; i > 0; --i) r[i] = (x > r[i - 1]) ? r[i - 1] : fmaxf(r[i], x);
    r[0] = fmaxf(r[0], x);
  }

  __device__ __forceinline__ void chunk(float (&v)[32], int col0) {
    if (col0 + 32 > p.V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j >= p.V) v[j] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (v[j] > r[kTopR - 1]) insert(v[j]);
  }

  template <int BN>
  __device__ __forceinline__ void tile(uint32_t taddr, int n, int) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; c += 2) {
      float v0[32], v1[32];
      tmem_ld32(taddr + c * 32, v0);
      tmem_ld32(taddr + c * 32 + 32, v1);
      tmem_wait_ld();
      pin(v0);
      pin(v1);
      chunk(v0, n * BN + c * 32);
      chunk(v1, n * BN + c * 32 + 32);
    }
  }

  __device__ __forceinline__ void end_unit(int split, int) {
    if (!row_ok) return;
    float4* o = reinterpret_cast<float4*>(p.topr + (static_cast<size_t>(split) * p.T + t) * kTopR);
    o[0] = make_float4(r[0], r[1], r[2], r[3]);
    o[1] = make_float4(r[4], r[5], r[6], r[7]);
  }
};

// ---------------------------------------------------------------- candidate pass epilogue
struct EpiCand {
  using Params = CandParams;
  const Params& p;
  int t;
  float th;

  __device__ explicit EpiCand(const Params& prm) : p(prm) {}

  __device__ __forceinline__ void begin_unit(int row0, int, int, int row) {
    t = row0 + row;
    th = t < p.T ? p.theta[t] : INFINITY;
  }

  __device__ __forceinline__ bool hit(float x, int col) const { return x >= th && col < p.V; }

  __device__ __forceinline__ int count(const float (&v)[32], int col0) const {
    int c = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) c += hit(v[j], col0 + j) ? 1 : 0;
    return c;
  }

  __device__ __forceinline__ void write(const float (&v)[32], int col0, int& pos) const {
    int2* row = p.cand + static_cast<size_t>(t) * p.cap;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (hit(v[j], col0 + j)) {
        if (pos < p.cap) row[pos] = make_int2(__float_as_int(v[j]), col0 + j);
        ++pos;
      }
    }
  }

  // Two passes over the tile's accumulator: count the row's candidates, claim their slots
  // with one atomic per row, then read the accumulator again and write them.  One atomic
  // round trip per tile instead of one per candidate column keeps the epilogue shorter than
  // the tile's MMAs.  tcgen05.ld is warp-collective, so both passes run on the whole warp.
  template <int BN>
  __device__ __forceinline__ void tile(uint32_t taddr, int n, int) {
    int total = 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; c += 2) {
      float v0[32], v1[32];
      tmem_ld32(taddr + c * 32, v0);
      tmem_ld32(taddr + c * 32 + 32, v1);
      tmem_wait_ld();
      pin(v0);
      pin(v1);
      total += count(v0, n * BN + c * 32) + count(v1, n * BN + c * 32 + 32);
    }
    if (!__any_sync(0xffffffffu, total > 0)) return;
    int pos = total > 0 ? atomicAdd(&p.cnt[t], total) : 0;
#pragma unroll 1
    for (int c = 0; c < BN / 32; c += 2) {
      float v0[32], v1[32];
      tmem_ld32(taddr + c * 32, v0);
      tmem_ld32(taddr + c * 32 + 32, v1);
      tmem_wait_ld();
      pin(v0);
      pin(v1);
      if (total > 0) {
        write(v0, n * BN + c * 32, pos);
        write(v1, n * BN + c * 32 + 32, pos);
      }
    }
  }

  __device__ __forceinline__ void end_unit(int, int) {}
};

// ---------------------------------------------------------------- bound and select kernels
// Orderable key: ascending key = logit descending, then id ascending.
__device__ __forceinline__ unsigned long long rank_key(float v, int id) {
  uint32_t b = __float_as_uint(v);
  b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);  // ascending float order as unsigned
  return (static_cast<unsigned long long>(~b) << 32) | static_cast<uint32_t>(id);
}

constexpr int kBoundWarps = 8;

// theta_t = the K-th largest of the row's S * kTopR kept logits (-inf when fewer than K).
__global__ void __launch_bounds__(kBoundWarps * 32)
    bound_kernel(const float* __restrict__ topr, int nsplit, int64_t T, int K, float* __restrict__ theta) {
  __shared__ float sv[kBoundWarps][kMaxBoundSplits * kTopR];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kBoundWarps + w;
  if (t >= T) return;  // uniform per warp
  const int n = nsplit * kTopR;
  for (int i = lane; i < n; i += 32) {
    const int s = i / kTopR, k = i - s * kTopR;
    sv[w][i] = topr[(static_cast<size_t>(s) * T + t) * kTopR + k];
  }
  __syncwarp();
  float th = -INFINITY;
  if (n >= K) {
    for (int i = lane; i < n; i += 32) {
      const float x = sv[w][i];
      int rank = 0;  // position of (x, i) in the order by value descending, then index
      for (int j = 0; j < n; ++j) {
        const float y = sv[w][j];
        rank += (y > x) || (y == x && j < i);
      }
      if (rank == K - 1) th = x;
    }
    th = fmaxf(th, __shfl_xor_sync(0xffffffffu, th, 16));
    th = fmaxf(th, __shfl_xor_sync(0xffffffffu, th, 8));
    th = fmaxf(th, __shfl_xor_sync(0xffffffffu, th, 4));
    th = fmaxf(th, __shfl_xor_sync(0xffffffffu, th, 2));
    th = fmaxf(th, __shfl_xor_sync(0xffffffffu, th, 1));
  }
  if (lane == 0) theta[t] = th;
}

constexpr int kSelectThreads = 256;

// Inverse of rank_key's logit part.
__device__ __forceinline__ float key_logit(unsigned long long key) {
  const uint32_t b = ~static_cast<uint32_t>(key >> 32);
  return __uint_as_float((b & 0x80000000u) ? (b & 0x7fffffffu) : ~b);
}

// One block per row: sorts the row's candidate keys in shared memory with a bitonic network
// (padded to a power of two with the largest key, which no candidate has) and writes the
// first K in order.
__global__ void __launch_bounds__(kSelectThreads)
    select_kernel(const int2* __restrict__ cand, const int* __restrict__ cnt, int cap, int K, int64_t T,
                  int32_t* __restrict__ out_idx, float* __restrict__ out_val, uint32_t* __restrict__ status) {
  extern __shared__ unsigned long long keys[];
  const int64_t t = blockIdx.x;
  if (t >= T) return;
  const int total = cnt[t];
  int32_t* oi = out_idx + t * K;
  float* ov = out_val + t * K;
  if (total > cap || total < K) {
    for (int k = threadIdx.x; k < K; k += kSelectThreads) {
      oi[k] = -1;
      ov[k] = NAN;
    }
    if (threadIdx.x == 0) atomicOr(status, kStatusTopkOverflowBit);
    return;
  }
  const int2* c = cand + t * cap;
  int n = 1;
  while (n < total) n <<= 1;
  for (int i = threadIdx.x; i < n; i += kSelectThreads)
    keys[i] = i < total ? rank_key(__int_as_float(c[i].x), c[i].y) : ~0ull;
  __syncthreads();
  // each step visits the n / 2 compare-exchange pairs (i, i + j) directly
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int q = threadIdx.x; q < n / 2; q += kSelectThreads) {
        const int i = 2 * q - (q & (j - 1));
        const int l = i + j;
        const unsigned long long a = keys[i], b = keys[l];
        if ((a > b) == ((i & k) == 0)) {
          keys[i] = b;
          keys[l] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int k = threadIdx.x; k < K; k += kSelectThreads) {
    const unsigned long long key = keys[k];
    oi[k] = static_cast<int32_t>(static_cast<uint32_t>(key));
    ov[k] = key_logit(key);
  }
}

__global__ void fill_kernel(float* __restrict__ a, int64_t n, float v) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) a[i] = v;
}

// ---------------------------------------------------------------- planning
struct TopkPlan {
  bool bound_pass;
  int stride;      // bound pass: every stride-th vocabulary row
  int64_t Vs;      // bound pass: rows it reads, ceil(V / stride)
  int cap;
  size_t off_topr, off_theta, off_cnt, off_cand, total;
};

// Values the bound pass keeps for a row over n vocabulary rows: kTopR per split.
static int64_t kept_values(int64_t n) {
  const int64_t tiles = (n + kVocabTile - 1) / kVocabTile;
  return (tiles < kMaxBoundSplits ? tiles : kMaxBoundSplits) * kTopR;
}

// max_stride: the largest sampling stride of the bound pass the caller allows (1, 2, 4 or 8).
static bool make_topk_plan(int64_t T, int64_t d, int64_t V, int64_t K, TopkPlan* p, int max_stride = kMaxBoundStride) {
  if (T < 0 || T >= (int64_t{1} << 31) || d < 8 || d % 8 != 0 || d >= (int64_t{1} << 20)) return false;
  if (V < 1 || V > (int64_t{1} << 30) || K < 1 || K > V) return false;
  p->bound_pass = V > kAllCandidatesV;
  p->stride = 1;
  p->Vs = V;
  if (p->bound_pass) {
    if (kept_values(V) < K) return false;
    while (p->stride < max_stride && kept_values((V + 2 * p->stride - 1) / (2 * p->stride)) >= K) p->stride *= 2;
    p->Vs = (V + p->stride - 1) / p->stride;
  }
  const int64_t cap = 4 * K * p->stride;
  p->cap = p->bound_pass ? static_cast<int>(cap > 512 ? cap : 512) : static_cast<int>(V);
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  size_t off = 256;  // status header
  p->off_topr = off;  off = up(off + static_cast<size_t>(T) * (p->bound_pass ? kMaxBoundSplits * kTopR * 4 : 0));
  p->off_theta = off; off = up(off + static_cast<size_t>(T) * 4);
  p->off_cnt = off;   off = up(off + static_cast<size_t>(T) * 4);
  p->off_cand = off;  off = up(off + static_cast<size_t>(T) * p->cap * 8);
  p->total = off;
  return true;
}

static fkl_status topk_fail(fkl_status s, const char* msg) {
  set_last_error_message(msg);
  return s;
}

}  // namespace fkl

using namespace fkl;

extern "C" size_t fkl_teacher_topk_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K) {
  TopkPlan p;
  return make_topk_plan(T, d, V, K, &p) ? p.total : 0;
}

extern "C" fkl_status fkl_teacher_topk(const uint16_t* Ht, const uint16_t* Wt, int64_t T, int64_t d, int64_t V,
                                       int64_t K, int32_t* topk_idx, float* topk_logits, void* workspace,
                                       size_t ws_bytes, void* stream) {
  return fkl_teacher_topk_ex(Ht, Wt, T, d, V, K, 0, topk_idx, topk_logits, workspace, ws_bytes, stream);
}

extern "C" fkl_status fkl_teacher_topk_ex(const uint16_t* Ht, const uint16_t* Wt, int64_t T, int64_t d, int64_t V,
                                          int64_t K, int32_t max_bound_stride, int32_t* topk_idx, float* topk_logits,
                                          void* workspace, size_t ws_bytes, void* stream) {
  set_last_error_message("");
  if (max_bound_stride != 0 && max_bound_stride != 1 && max_bound_stride != 2 && max_bound_stride != 4 &&
      max_bound_stride != 8)
    return topk_fail(FKL_ERR_INVALID_ARG, "max_bound_stride must be 0 (default), 1, 2, 4 or 8");
  TopkPlan pl;
  if (!make_topk_plan(T, d, V, K, &pl, max_bound_stride == 0 ? kMaxBoundStride : max_bound_stride))
    return topk_fail(FKL_ERR_INVALID_ARG,
                     "unsupported shape (need d % 8 == 0, 1 <= K <= V, and K <= 256 with K <= 8 * ceil(V / 256) "
                     "when V > 4096)");
  if (Wt == nullptr || (T > 0 && (Ht == nullptr || topk_idx == nullptr || topk_logits == nullptr)))
    return topk_fail(FKL_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((reinterpret_cast<uintptr_t>(Ht) | reinterpret_cast<uintptr_t>(Wt)) % 16 != 0 ||
      (reinterpret_cast<uintptr_t>(topk_idx) | reinterpret_cast<uintptr_t>(topk_logits)) % 4 != 0)
    return topk_fail(FKL_ERR_ALIGNMENT, "Ht and Wt need 16-byte alignment, the outputs 4-byte");
  if (workspace == nullptr || ws_bytes < pl.total) return topk_fail(FKL_ERR_WORKSPACE, "workspace missing or too small");
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return topk_fail(FKL_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return topk_fail(FKL_ERR_CUDA, "device query failed");
  if (major != 10 || minor != 3) return topk_fail(FKL_ERR_UNSUPPORTED, "device is not sm_103");
  {
    const NamedPtr ptrs[] = {{Ht, "Ht"}, {Wt, "Wt"}, {topk_idx, "topk_idx"}, {topk_logits, "topk_logits"},
                             {workspace, "workspace"}};
    const int s = check_device_memory(ptrs);
    if (s != FKL_OK) return static_cast<fkl_status>(s);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  int* items_taken = reinterpret_cast<int*>(ws + 16);  // work-item counter of both passes
  int sched_base = 0;
  if (cudaMemsetAsync(ws, 0, 256, st) != cudaSuccess) return topk_fail(FKL_ERR_CUDA, "cudaMemsetAsync failed");
  if (T == 0) return FKL_OK;
  float* topr = reinterpret_cast<float*>(ws + pl.off_topr);
  float* theta = reinterpret_cast<float*>(ws + pl.off_theta);
  int* cnt = reinterpret_cast<int*>(ws + pl.off_cnt);
  int2* cand = reinterpret_cast<int2*>(ws + pl.off_cand);
  if (cudaMemsetAsync(cnt, 0, static_cast<size_t>(T) * 4, st) != cudaSuccess)
    return topk_fail(FKL_ERR_CUDA, "cudaMemsetAsync failed");

  CUtensorMap mH, mW, mWs;
  if (!encode_map_bf16(&mH, Ht, d, T, d * 2, 64, 128) || !encode_map_bf16(&mW, Wt, d, V, d * 2, 64, kVocabTile / 2) ||
      !encode_map_bf16(&mWs, Wt, d, pl.Vs, d * 2 * pl.stride, 64, kVocabTile / 2))
    return topk_fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed");
  const int m_tiles = static_cast<int>((T + 255) / 256), n_tiles = static_cast<int>((V + kVocabTile - 1) / kVocabTile);
  if (pl.bound_pass) {
    const int s_tiles = static_cast<int>((pl.Vs + kVocabTile - 1) / kVocabTile);
    const int ns = s_tiles < kMaxBoundSplits ? s_tiles : kMaxBoundSplits;
    GemmShape g = make_shape(T, pl.Vs, d, kVocabTile, ns, status, 256);
    g.group_m = group_rows(g.m_tiles);
    g.sched = items_taken;  // units drawn from the counter (zeroed with the header)
    sched_base = num_items(g);
    TopRParams tp;
    tp.topr = topr;
    tp.T = static_cast<int>(T);
    tp.V = static_cast<int>(pl.Vs);
    trace_launch_begin(st);
    if (launch_gemm2_t<kVocabTile, false, false, EpiTopR>(mH, mWs, g, tp, sms, st) != cudaSuccess)
      return topk_fail(FKL_ERR_CUDA, "bound-pass GEMM launch failed");
    trace_launch_end(st, 5, 2.0 * T * pl.Vs * d);
    bound_kernel<<<static_cast<unsigned>((T + kBoundWarps - 1) / kBoundWarps), kBoundWarps * 32, 0, st>>>(
        topr, ns, T, static_cast<int>(K), theta);
  } else {
    fill_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, st>>>(theta, T, -INFINITY);
  }
  if (cudaGetLastError() != cudaSuccess) return topk_fail(FKL_ERR_CUDA, "bound kernel launch failed");
  GemmShape g2 = make_shape(T, V, d, kVocabTile, dynamic_splits(m_tiles, n_tiles, sms / 2), status, 256);
  g2.group_m = group_rows(g2.m_tiles);
  g2.sched = items_taken;  // after the bound pass's items, if it ran
  g2.sched_base = sched_base;
  CandParams cp;
  cp.theta = theta;
  cp.cnt = cnt;
  cp.cand = cand;
  cp.cap = pl.cap;
  cp.T = static_cast<int>(T);
  cp.V = static_cast<int>(V);
  trace_launch_begin(st);
  if (launch_gemm2_t<kVocabTile, false, false, EpiCand>(mH, mW, g2, cp, sms, st) != cudaSuccess)
    return topk_fail(FKL_ERR_CUDA, "candidate-pass GEMM launch failed");
  trace_launch_end(st, 6, 2.0 * T * V * d);
  size_t pow2 = 1;
  while (pow2 < static_cast<size_t>(pl.cap)) pow2 <<= 1;
  const size_t smem = pow2 * 8;  // the bitonic sort's keys, padded to a power of two
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return topk_fail(FKL_ERR_CUDA, "cudaFuncSetAttribute failed");
  select_kernel<<<static_cast<unsigned>(T), kSelectThreads, smem, st>>>(cand, cnt, pl.cap, static_cast<int>(K), T,
                                                                       topk_idx, topk_logits, status);
  if (cudaGetLastError() != cudaSuccess) return topk_fail(FKL_ERR_CUDA, "select kernel launch failed");
  return FKL_OK;
}
