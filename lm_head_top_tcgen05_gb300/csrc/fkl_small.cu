// The light kernels around the tensor-core GEMMs:
//   prep      teacher side of the loss: p = softmax(z / tau) over the K cached slots,
//             c_t = sum_k p log p, and the (id, p) pairs of each row sorted by id so that
//             the GEMM epilogues can walk them in step with the vocabulary tiles;
//   weights   the weight w_t of each token's KL in the loss: 1/N (token mean) or
//             1/(S N_s) (mean over the S packed sequences of each sequence's token mean),
//             0 for masked tokens; from integer counts, so deterministic;
//   combine   merges the forward's per-split partials into lse_t and KL_t and reduces
//             sum_t w_t KL_t in a fixed order (no float atomics: deterministic);
//   scalars   g * tau for the backward's dS scale (g may live on the device);
//   poison    fills the gradients with NaN when the device recorded an error;
//   timeout   one bounded wait that nothing completes (checks the timeout path).
#include <climits>
#include <cmath>

#include "fkl_ptx.cuh"

namespace fkl {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kPrepWarps = 8;

// One warp per token row.  The row's K ids and logits are read with coalesced loads
// (consecutive lanes, consecutive slots); ids are staged in shared memory to rank them.
__global__ void __launch_bounds__(kPrepWarps * 32)
    prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ z, int64_t T, int K, int V,
                float inv_tau, int2* __restrict__ pairs, float* __restrict__ crow,
                uint32_t* __restrict__ status) {
  extern __shared__ int sid[];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kPrepWarps + w;
  if (t >= T) return;  // uniform per warp
  int* my = sid + w * K;
  const int32_t* ri = idx + t * K;
  const float* rz = z + t * K;

  uint32_t bad = 0;
  float zmax = -INFINITY;
  for (int k = lane; k < K; k += 32) {
    int id = ri[k];
    if (id < 0 || id >= V) {
      bad |= kStatusBadIdBit;
      id = INT_MAX;  // never matches a column; sorts last
    } else {
      zmax = fmaxf(zmax, rz[k] * inv_tau);
    }
    my[k] = id;
  }
  zmax = warp_max(zmax);
  const bool row_ok = zmax > -INFINITY;
  float Z = 0.f;
  if (row_ok) {
    for (int k = lane; k < K; k += 32)
      if (my[k] != INT_MAX) Z += expf(rz[k] * inv_tau - zmax);
  }
  Z = warp_sum(Z);
  const float logZ = row_ok ? logf(Z) : 0.f;
  __syncwarp();
  float c = 0.f;
  for (int k = lane; k < K; k += 32) {
    const int id = my[k];
    float pk = 0.f;
    if (row_ok && id != INT_MAX) {
      const float zz = rz[k] * inv_tau;
      if (zz > -INFINITY) {
        const float lp = (zz - zmax) - logZ;
        pk = expf(lp);
        c = fmaf(pk, lp, c);
      }
    }
    int rank = 0;  // position of (id, k) in the order by id, then slot
    for (int j = 0; j < K; ++j) {
      const int o = my[j];
      rank += (o < id) || (o == id && j < k);
    }
    pairs[t * K + rank] = make_int2(id, __float_as_int(pk));
  }
  c = warp_sum(c);
  if (!row_ok) bad |= kStatusBadRowBit;
  bad = __reduce_or_sync(0xffffffffu, bad);
  if (lane == 0) {
    crow[t] = row_ok ? c : 0.f;
    if (bad) atomicOr(status, bad);
  }
}

cudaError_t launch_prep(const int32_t* idx, const float* logits, int64_t T, int K, int V, float tau,
                        int2* pairs, float* crow, uint32_t* status, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kPrepWarps) * K * sizeof(int);
  const int64_t blocks = (T + kPrepWarps - 1) / kPrepWarps;
  prep_kernel<<<static_cast<unsigned>(blocks), kPrepWarps * 32, smem, st>>>(
      idx, logits, T, K, V, 1.0f / tau, pairs, crow, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine
constexpr int kCombineThreads = 256;

// Per token: lse_t from the splits' (max, sum) in base 2, KL_t = c_t - g_t / tau + lse_t,
// then a fixed-order tree sum of w_t KL_t over the tokens of the block.
__global__ void __launch_bounds__(kCombineThreads)
    combine_rows_kernel(const float* __restrict__ part, int nsplit, const float* __restrict__ crow,
                        const float* __restrict__ wrow, int64_t T, float inv_tau,
                        float* __restrict__ lse, double* __restrict__ bsum, int* __restrict__ bcnt) {
  __shared__ double ssum[kCombineThreads];
  __shared__ int scnt[kCombineThreads];
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x;
  double kl = 0.0;
  int cnt = 0;
  if (t < T) {
    const size_t plane = static_cast<size_t>(nsplit) * T;
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part[static_cast<size_t>(s) * T + t]);
    float L = 0.f, G = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t i = static_cast<size_t>(s) * T + t;
      L += part[plane + i] * exp2f(part[i] - M);
      G += part[2 * plane + i];
    }
    const float lse_t = (M + log2f(L)) * 0.69314718055994531f;
    lse[t] = lse_t;
    const float w = wrow[t];
    if (w != 0.f) {
      kl = static_cast<double>(w) *
           (static_cast<double>(crow[t]) - static_cast<double>(G) * inv_tau + static_cast<double>(lse_t));
      cnt = 1;
    }
  }
  ssum[threadIdx.x] = kl;
  scnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = kCombineThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    bsum[blockIdx.x] = ssum[0];
    bcnt[blockIdx.x] = scnt[0];
  }
}

constexpr int kFinalThreads = 1024;

__global__ void __launch_bounds__(kFinalThreads)
    combine_final_kernel(const double* __restrict__ bsum, const int* __restrict__ bcnt, int64_t nb,
                         float tau, WsHeader* hdr, float* loss) {
  __shared__ double ssum[kFinalThreads];
  __shared__ long long scnt[kFinalThreads];
  double s = 0.0;
  long long c = 0;
  for (int64_t i = threadIdx.x; i < nb; i += kFinalThreads) {
    s += bsum[i];
    c += bcnt[i];
  }
  ssum[threadIdx.x] = s;
  scnt[threadIdx.x] = c;
  __syncthreads();
  for (int o = kFinalThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      ssum[threadIdx.x] += ssum[threadIdx.x + o];
      scnt[threadIdx.x] += scnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double L = scnt[0] > 0 ? static_cast<double>(tau) * tau * ssum[0] : 0.0;
    if (hdr->status != 0u) L = NAN;
    *loss = static_cast<float>(L);
  }
}

cudaError_t launch_combine(const float* part, int nsplit, const float* crow, const float* wrow,
                           int64_t T, float tau, float* lse, double* bsum, int* bcnt, int64_t nb,
                           WsHeader* hdr, float* loss, cudaStream_t st) {
  if (T > 0) {
    combine_rows_kernel<<<static_cast<unsigned>(nb), kCombineThreads, 0, st>>>(
        part, nsplit, crow, wrow, T, 1.0f / tau, lse, bsum, bcnt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  combine_final_kernel<<<1, kFinalThreads, 0, st>>>(bsum, bcnt, T > 0 ? nb : 0, tau, hdr, loss);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- token weights
constexpr int kWeightThreads = 256;

// Valid tokens per sequence (token mean: everything in sequence 0).  Integer atomics: the
// counts do not depend on the order of the additions.
__global__ void __launch_bounds__(kWeightThreads)
    seq_count_kernel(const uint8_t* __restrict__ mask, const int32_t* __restrict__ seq, int64_t T,
                     int num_seqs, int* __restrict__ cnt, uint32_t* __restrict__ status) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWeightThreads + threadIdx.x;
  if (t >= T) return;
  if (mask != nullptr && mask[t] == 0) return;
  const int sid = seq ? seq[t] : 0;
  if (sid < 0 || sid >= num_seqs) {
    atomicOr(status, kStatusBadSeqBit);
    return;
  }
  atomicAdd(&cnt[sid], 1);
}

// N = sum of the counts, S = number of sequences with a valid token (fixed-order tree sums).
__global__ void __launch_bounds__(kFinalThreads)
    seq_total_kernel(const int* __restrict__ cnt, int num_seqs, WsHeader* hdr) {
  __shared__ long long sn[kFinalThreads];
  __shared__ int ss[kFinalThreads];
  long long n = 0;
  int nz = 0;
  for (int i = threadIdx.x; i < num_seqs; i += kFinalThreads) {
    n += cnt[i];
    nz += cnt[i] > 0;
  }
  sn[threadIdx.x] = n;
  ss[threadIdx.x] = nz;
  __syncthreads();
  for (int o = kFinalThreads / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      sn[threadIdx.x] += sn[threadIdx.x + o];
      ss[threadIdx.x] += ss[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    hdr->n_valid = static_cast<int32_t>(sn[0]);
    hdr->n_seqs = ss[0];
  }
}

__global__ void __launch_bounds__(kWeightThreads)
    row_weight_kernel(const uint8_t* __restrict__ mask, const int32_t* __restrict__ seq, int64_t T,
                      int num_seqs, int per_sequence, const int* __restrict__ cnt, const WsHeader* hdr,
                      float* __restrict__ wrow) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWeightThreads + threadIdx.x;
  if (t >= T) return;
  float w = 0.f;
  const bool valid = mask == nullptr || mask[t] != 0;
  const int sid = seq ? seq[t] : 0;
  if (valid && sid >= 0 && sid < num_seqs) {
    if (per_sequence) {
      w = static_cast<float>(1.0 / (static_cast<double>(hdr->n_seqs) * static_cast<double>(cnt[sid])));
    } else {
      w = static_cast<float>(1.0 / static_cast<double>(hdr->n_valid));
    }
  }
  wrow[t] = w;
}

cudaError_t launch_weights(const uint8_t* mask, const int32_t* seq, int num_seqs, int per_sequence,
                           int64_t T, int* cnt, WsHeader* hdr, float* wrow, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(num_seqs) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((T + kWeightThreads - 1) / kWeightThreads);
  seq_count_kernel<<<blocks, kWeightThreads, 0, st>>>(mask, seq, T, num_seqs, cnt, &hdr->status);
  seq_total_kernel<<<1, kFinalThreads, 0, st>>>(cnt, num_seqs, hdr);
  row_weight_kernel<<<blocks, kWeightThreads, 0, st>>>(mask, seq, T, num_seqs, per_sequence, cnt, hdr, wrow);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- backward scale
__global__ void grad_scale_kernel(const float* grad, float tau, WsHeader* hdr) {
  hdr->gtau = (grad ? *grad : 1.0f) * tau;
}

cudaError_t launch_grad_scale(const float* grad, float tau, WsHeader* hdr, cudaStream_t st) {
  grad_scale_kernel<<<1, 1, 0, st>>>(grad, tau, hdr);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- poison on error
__global__ void poison_kernel(float* a, int64_t na, float* b, int64_t nb, const uint32_t* status) {
  if (*reinterpret_cast<const volatile uint32_t*>(status) == 0u) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na; i += stride) a[i] = NAN;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nb; i += stride) b[i] = NAN;
}

cudaError_t launch_poison(float* a, int64_t na, float* b, int64_t nb, const uint32_t* status,
                          int sms, cudaStream_t st) {
  poison_kernel<<<sms * 4, 256, 0, st>>>(a, na, b, nb, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- timeout probe
__global__ void wait_timeout_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtl ctl{&abort_flag, status, limit_ns};
    mbar_wait(b, 0u, ctl);  // nothing arrives: runs out after limit_ns
  }
}

cudaError_t launch_wait_timeout_test(uint32_t* status, uint64_t limit_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace fkl
