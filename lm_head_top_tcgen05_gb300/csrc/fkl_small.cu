// The light kernels around the tensor-core GEMMs:
//   prep      teacher side of the loss: p = softmax(z / tau) over the K cached slots,
//             c_t = sum_k p log p, and the (id, p) pairs of each row sorted by id so that
//             the GEMM epilogues can walk them in step with the vocabulary tiles;
//   weights   the weight w_t of each token's KL in the loss: 1/N (token mean) or
//             1/(S N_s) (mean over the S packed sequences of each sequence's token mean),
//             0 for masked tokens, with N or S the whole batch's when the batch is split
//             over several calls; from integer counts, so deterministic;
//   combine   merges the forward's per-split partials into lse_t and KL_t and reduces
//             sum_t w_t KL_t in a fixed order (no float atomics: deterministic);
//   div       the other divergences: D_t from the student logits at the cached ids
//             (forward) and the per-row / per-id terms of their dS (backward);
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
constexpr int kSortMaxK = 128;  // up to this K a row's pairs are sorted in registers

// Teacher side of one row from its valid slots: log Z over the tempered logits (zz = z / tau,
// -inf for ids outside [0, V)), then p_k = exp(zz_k - zmax - log Z) and c += p_k log p_k.
__device__ __forceinline__ float teacher_p(float zz, bool valid, float zmax, float logZ, float& c) {
  if (!valid || !(zz > -INFINITY)) return 0.f;
  const float lp = (zz - zmax) - logZ;
  const float pk = expf(lp);
  c = fmaf(pk, lp, c);
  return pk;
}

// Sorts 128 keys held 4 per lane (element i = e * 32 + lane in keys[e]) ascending: a bitonic
// network, exchanging across lanes by shuffles for distances below 32 and inside the lane's
// registers for 32 and 64.
__device__ __forceinline__ void warp_sort128(unsigned long long (&keys)[4], int lane) {
#pragma unroll
  for (int k = 2; k <= 128; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int je = j >> 5;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e & je) continue;
          const int e2 = e | je;
          const bool asc = (((e << 5) | lane) & k) == 0;
          const unsigned long long a = keys[e], b = keys[e2];
          const unsigned long long lo = a < b ? a : b, hi = a < b ? b : a;
          keys[e] = asc ? lo : hi;
          keys[e2] = asc ? hi : lo;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, keys[e], j);
          const bool asc = (((e << 5) | lane) & k) == 0;
          const bool lower = (lane & j) == 0;
          const unsigned long long a = keys[e];
          keys[e] = (asc == lower) ? (a < o ? a : o) : (a < o ? o : a);
        }
      }
    }
  }
}

// One warp per token row.  The row's K ids and logits are read with coalesced loads
// (consecutive lanes, consecutive slots).  The (id, slot) pairs are ordered by id, then
// slot: for K <= 128 by a register bitonic sort of 64-bit keys (id << 32 | slot), otherwise
// by ranking each pair against the row's ids staged in shared memory.  Both give the same
// order.
__global__ void __launch_bounds__(kPrepWarps * 32)
    prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ z, int64_t T, int K, int V,
                float inv_tau, int2* __restrict__ pairs, int* __restrict__ slot, float* __restrict__ crow,
                uint32_t* __restrict__ status) {
  extern __shared__ int sid[];  // [kPrepWarps][K]: p by slot (sort path) or ids (rank path)
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kPrepWarps + w;
  if (t >= T) return;  // uniform per warp
  int* my = sid + w * K;
  const int32_t* ri = idx + t * K;
  const float* rz = z + t * K;
  uint32_t bad = 0;
  float c = 0.f;
  bool row_ok;

  if (K <= kSortMaxK) {
    int id[4];
    float zz[4];
    float zmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = (e << 5) | lane;
      id[e] = INT_MAX;
      zz[e] = -INFINITY;
      if (k < K) {
        const int v = ri[k];
        if (v < 0 || v >= V) {
          bad |= kStatusBadIdBit;  // INT_MAX never matches a column and sorts last
        } else {
          id[e] = v;
          zz[e] = rz[k] * inv_tau;
          zmax = fmaxf(zmax, zz[e]);
        }
      }
    }
    zmax = warp_max(zmax);
    row_ok = zmax > -INFINITY;
    float Z = 0.f;
    if (row_ok) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (id[e] != INT_MAX) Z += expf(zz[e] - zmax);
    }
    Z = warp_sum(Z);
    const float logZ = row_ok ? logf(Z) : 0.f;
    float* sp = reinterpret_cast<float*>(my);
    unsigned long long keys[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = (e << 5) | lane;
      keys[e] = ~0ull;  // padding sorts after every slot
      if (k < K) {
        sp[k] = teacher_p(zz[e], row_ok && id[e] != INT_MAX, zmax, logZ, c);
        keys[e] = (static_cast<unsigned long long>(static_cast<uint32_t>(id[e])) << 32) | static_cast<uint32_t>(k);
      }
    }
    warp_sort128(keys, lane);
    __syncwarp();
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = (e << 5) | lane;
      if (i < K) {
        const int k = static_cast<int>(keys[e] & 0xffffffffull);
        pairs[t * K + i] = make_int2(static_cast<int>(keys[e] >> 32), __float_as_int(sp[k]));
        if (slot) slot[t * K + i] = k;
      }
    }
  } else {
    float zmax = -INFINITY;
    for (int k = lane; k < K; k += 32) {
      int v = ri[k];
      if (v < 0 || v >= V) {
        bad |= kStatusBadIdBit;
        v = INT_MAX;
      } else {
        zmax = fmaxf(zmax, rz[k] * inv_tau);
      }
      my[k] = v;
    }
    zmax = warp_max(zmax);
    row_ok = zmax > -INFINITY;
    float Z = 0.f;
    if (row_ok) {
      for (int k = lane; k < K; k += 32)
        if (my[k] != INT_MAX) Z += expf(rz[k] * inv_tau - zmax);
    }
    Z = warp_sum(Z);
    const float logZ = row_ok ? logf(Z) : 0.f;
    __syncwarp();
    for (int k = lane; k < K; k += 32) {
      const int v = my[k];
      const float pk = teacher_p(rz[k] * inv_tau, row_ok && v != INT_MAX, zmax, logZ, c);
      int rank = 0;  // position of (id, k) in the order by id, then slot
      for (int j = 0; j < K; ++j) {
        const int o = my[j];
        rank += (o < v) || (o == v && j < k);
      }
      pairs[t * K + rank] = make_int2(v, __float_as_int(pk));
      if (slot) slot[t * K + rank] = k;
    }
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
                        int2* pairs, int* slot, float* crow, uint32_t* status, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kPrepWarps) * K * sizeof(int);
  const int64_t blocks = (T + kPrepWarps - 1) / kPrepWarps;
  prep_kernel<<<static_cast<unsigned>(blocks), kPrepWarps * 32, smem, st>>>(
      idx, logits, T, K, V, 1.0f / tau, pairs, slot, crow, status);
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
    const float lse_t = (M + log2f(L)) * kLn2;
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

cudaError_t launch_combine_rows(const float* part, int nsplit, const float* crow, const float* wrow,
                                int64_t T, float tau, float* lse, double* bsum, int* bcnt, int64_t nb,
                                cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  combine_rows_kernel<<<static_cast<unsigned>(nb), kCombineThreads, 0, st>>>(
      part, nsplit, crow, wrow, T, 1.0f / tau, lse, bsum, bcnt);
  return cudaGetLastError();
}

cudaError_t launch_combine_final(const double* bsum, const int* bcnt, int64_t T, int64_t nb, float tau,
                                 WsHeader* hdr, float* loss, cudaStream_t st) {
  combine_final_kernel<<<1, kFinalThreads, 0, st>>>(bsum, bcnt, T > 0 ? nb : 0, tau, hdr, loss);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* part, int nsplit, const float* crow, const float* wrow,
                           int64_t T, float tau, float* lse, double* bsum, int* bcnt, int64_t nb,
                           WsHeader* hdr, float* loss, cudaStream_t st) {
  cudaError_t e = launch_combine_rows(part, nsplit, crow, wrow, T, tau, lse, bsum, bcnt, nb, st);
  if (e != cudaSuccess) return e;
  return launch_combine_final(bsum, bcnt, T, nb, tau, hdr, loss, st);
}

// ---------------------------------------------------------------- other divergences
// With p the teacher's probability at one id (its slots added), q = exp(s / tau - lse) the
// student's and D = sum over the row's ids of phi(p, q) + psi * (student mass outside
// them), the per-id terms are phi and q * gamma, gamma = dD/dq at that id (psi outside).
// Written out per divergence from its definition (JSD: m = b p + (1 - b) q; skew KL:
// m = a p + (1 - a) q; skew reverse KL: m = a q + (1 - a) p):
//   JSD        phi = b p log(p / m) + (1 - b) q log(q / m)   q gamma = (1 - b) q log(q / m)
//              psi = -(1 - b) log(1 - b)
//   skew KL    phi = p log(p / m)                            q gamma = -(1 - a) p q / m
//              psi = 0
//   skew RKL   phi = q log(q / m)                            q gamma = q (log(q / m) + 1 - a q / m)
//              psi = -log a
//   TV         phi = |p - q| / 2                             q gamma = -q sign(p - q) / 2
//              psi = 1 / 2
// log q is taken as s / tau - lse, so the terms stay finite where q underflows.
__device__ __forceinline__ float div_psi(const DivSpec& dv) {
  switch (dv.kind) {
    case 1: return -(1.f - dv.param) * log1pf(-dv.param);
    case 3: return -logf(dv.param);
    case 4: return 0.5f;
    default: return 0.f;
  }
}

__device__ __forceinline__ void div_terms(const DivSpec& dv, float p, float logq, float& phi, float& qg) {
  const float q = expf(logq);
  const float c = dv.param;
  switch (dv.kind) {
    case 1: {
      const float lm = logf(fmaf(c, p, (1.f - c) * q));
      const float ql = q * (logq - lm);
      phi = c * p * (logf(p) - lm) + (1.f - c) * ql;
      qg = (1.f - c) * ql;
      break;
    }
    case 2: {
      const float m = fmaf(c, p, (1.f - c) * q);
      const float lm = c == 0.f ? logq : logf(m);
      phi = p * (logf(p) - lm);
      qg = -(1.f - c) * p * (c == 0.f ? 1.f : q / m);
      break;
    }
    case 3: {
      if (c == 1.f) { phi = 0.f; qg = 0.f; break; }
      const float m = fmaf(c, q, (1.f - c) * p);
      const float l = logq - logf(m);
      phi = q * l;
      qg = q * (l + 1.f - c * q / m);
      break;
    }
    case 4: {
      const float dlt = p - q;
      phi = 0.5f * fabsf(dlt);
      qg = dlt > 0.f ? -0.5f * q : (dlt < 0.f ? 0.5f * q : 0.f);
      break;
    }
    default: {  // KL
      phi = p * (logf(p) - logq);
      qg = -p;
    }
  }
}

// Per-row sums over the merged ids of one row (warp per row; lanes over sorted positions):
// phi, q and q * gamma.  The pair at position j starts a run of equal ids unless position
// j - 1 holds the same id; the run's first position carries the run's total p, the others
// contribute nothing.  Ids outside [0, V) (sorted last as INT_MAX) and p = 0 are skipped.
// s_at(j) gives the student logit at position j.  If r_out is not NULL, the per-position
// term r = q psi - q gamma (0 off a run start) is stored there, after the whole warp has
// read the row.
template <class SAt>
__device__ __forceinline__ void div_row(const DivSpec& dv, const int2* row, int K, float lse, float inv_tau,
                                        float psi, SAt s_at, int lane, float& sphi, float& sq, float& sqg,
                                        int2* r_out) {
  sphi = 0.f;
  sq = 0.f;
  sqg = 0.f;
  for (int j0 = 0; j0 < K; j0 += 32) {
    const int j = j0 + lane;
    float r = 0.f;
    if (j < K) {
      const int id = row[j].x;
      const bool start = id != INT_MAX && (j == 0 || row[j - 1].x != id);
      if (start) {
        float p = __int_as_float(row[j].y);
        for (int jj = j + 1; jj < K && row[jj].x == id; ++jj) p += __int_as_float(row[jj].y);
        if (p > 0.f) {
          const float logq = s_at(j) * inv_tau - lse;
          float phi, qg;
          div_terms(dv, p, logq, phi, qg);
          const float q = expf(logq);
          sphi += phi;
          sq += q;
          sqg += qg;
          r = q * psi - qg;
        }
      }
    }
    if (r_out) {
      __syncwarp();
      if (j < K) r_out[j].y = __float_as_int(r);
      __syncwarp();
    }
  }
  sphi = warp_sum(sphi);
  sq = warp_sum(sq);
  sqg = warp_sum(sqg);
}

constexpr int kDivRowsThreads = 256;  // 8 warps; a block covers the combine's 256-row block

__global__ void __launch_bounds__(kDivRowsThreads)
    div_rows_kernel(DivSpec dv, int compute, const int2* __restrict__ pairs, const int* __restrict__ slot,
                    const float* __restrict__ sg, const float* __restrict__ lse, const float* __restrict__ wrow,
                    int64_t T, int K, float inv_tau, float* __restrict__ user_s, double* __restrict__ bsum,
                    int* __restrict__ bcnt) {
  __shared__ double ssum[kDivRowsThreads];
  __shared__ int scnt[kDivRowsThreads];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float psi = div_psi(dv);
  for (int i = w; i < kDivRowsThreads; i += kDivRowsThreads / 32) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kDivRowsThreads + i;
    double v = 0.0;
    int c = 0;
    if (t < T) {
      const int2* row = pairs + t * K;
      const float* srow = sg + t * K;
      if (user_s) {
        for (int j = lane; j < K; j += 32)
          user_s[t * K + slot[t * K + j]] = row[j].x == INT_MAX ? NAN : srow[j];
      }
      const float wt = wrow[t];
      if (compute && wt != 0.f) {
        float sphi, sq, sqg;
        div_row(dv, row, K, lse[t], inv_tau, psi, [&](int j) { return srow[j]; }, lane, sphi, sq, sqg, nullptr);
        v = static_cast<double>(wt) * (static_cast<double>(sphi) + static_cast<double>(psi) * (1.0 - sq));
        c = 1;
      }
    }
    if (lane == 0) {
      ssum[i] = v;
      scnt[i] = c;
    }
  }
  if (!compute) return;
  __syncthreads();
  for (int o = kDivRowsThreads / 2; o > 0; o >>= 1) {
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

cudaError_t launch_div_rows(DivSpec dv, const int2* pairs, const int* slot, const float* sg,
                            const float* lse, const float* wrow, int64_t T, int K, float tau,
                            float* user_s, double* bsum, int* bcnt, int64_t nb, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int compute = dv.kind != 0;
  if (!compute && user_s == nullptr) return cudaSuccess;
  div_rows_kernel<<<static_cast<unsigned>(nb), kDivRowsThreads, 0, st>>>(
      dv, compute, pairs, slot, sg, lse, wrow, T, K, 1.0f / tau, user_s, bsum, bcnt);
  return cudaGetLastError();
}

constexpr int kDivCoefWarps = 8;

// a_t = psi - gbar, gbar = sum over ids of q gamma + psi (1 - sum over ids of q): then
// dD/ds_v = q_v (gamma_v - gbar) / tau = (a_t q_v - r_v) / tau with r = q psi - q gamma at
// the ids and 0 elsewhere (gamma = psi there).
__global__ void __launch_bounds__(kDivCoefWarps * 32)
    div_coef_kernel(DivSpec dv, int2* __restrict__ pairs, const int* __restrict__ slot,
                    const float* __restrict__ user_s, const float* __restrict__ lse, int64_t T, int K,
                    float inv_tau, float* __restrict__ arow) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kDivCoefWarps + w;
  if (t >= T) return;  // uniform per warp
  const float psi = div_psi(dv);
  int2* row = pairs + t * K;
  const int* srow = slot + t * K;
  const float* us = user_s + t * K;
  float sphi, sq, sqg;
  div_row(dv, row, K, lse[t], inv_tau, psi, [&](int j) { return us[srow[j]]; }, lane, sphi, sq, sqg, row);
  if (lane == 0) arow[t] = psi - (sqg + psi * (1.f - sq));
}

cudaError_t launch_div_coef(DivSpec dv, int2* pairs, const int* slot, const float* user_s,
                            const float* lse, int64_t T, int K, float tau, float* arow, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int64_t blocks = (T + kDivCoefWarps - 1) / kDivCoefWarps;
  div_coef_kernel<<<static_cast<unsigned>(blocks), kDivCoefWarps * 32, 0, st>>>(
      dv, pairs, slot, user_s, lse, T, K, 1.0f / tau, arow);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- token weights
constexpr int kWeightThreads = 256;

// Valid tokens per sequence (token mean: everything in sequence 0).  Integer atomics: the
// counts do not depend on the order of the additions.  The lanes of a warp that count into
// the same sequence add together (one atomic per sequence per warp instead of one per token,
// which for the token mean would serialise every token on one address).
__global__ void __launch_bounds__(kWeightThreads)
    seq_count_kernel(const uint8_t* __restrict__ mask, const int32_t* __restrict__ seq, int64_t T,
                     int num_seqs, int* __restrict__ cnt, uint32_t* __restrict__ status) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWeightThreads + threadIdx.x;
  int key = -1;  // the sequence this lane counts into, -1 for none
  if (t < T && (mask == nullptr || mask[t] != 0)) {
    const int sid = seq ? seq[t] : 0;
    if (sid < 0 || sid >= num_seqs) atomicOr(status, kStatusBadSeqBit);
    else key = sid;
  }
  const unsigned same = __match_any_sync(0xffffffffu, key);
  const int lane = threadIdx.x & 31;
  if (key >= 0 && lane == __ffs(same) - 1) atomicAdd(&cnt[key], __popc(same));
}

// N = sum of the counts, S = number of sequences with a valid token (fixed-order tree sums).
// With a global count (the whole batch's N, or S per_sequence), it must not be below this
// call's own.  count_out, if not NULL, receives this call's own count.
__global__ void __launch_bounds__(kFinalThreads)
    seq_total_kernel(const int* __restrict__ cnt, int num_seqs, int per_sequence,
                     const int64_t* __restrict__ global_count, WsHeader* hdr, int64_t* __restrict__ count_out) {
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
    const long long own = per_sequence ? ss[0] : sn[0];
    if (global_count != nullptr && *global_count < own) atomicOr(&hdr->status, kStatusBadCountBit);
    if (count_out != nullptr) *count_out = own;
  }
}

__global__ void __launch_bounds__(kWeightThreads)
    row_weight_kernel(const uint8_t* __restrict__ mask, const int32_t* __restrict__ seq, int64_t T,
                      int num_seqs, int per_sequence, const int* __restrict__ cnt, const WsHeader* hdr,
                      const int64_t* __restrict__ global_count, float* __restrict__ wrow) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWeightThreads + threadIdx.x;
  if (t >= T) return;
  float w = 0.f;
  const bool valid = mask == nullptr || mask[t] != 0;
  const int sid = seq ? seq[t] : 0;
  if (valid && sid >= 0 && sid < num_seqs) {
    // the mean's count: the whole batch's when given, else this call's own
    const double count = global_count != nullptr ? static_cast<double>(*global_count)
                                                 : static_cast<double>(per_sequence ? hdr->n_seqs : hdr->n_valid);
    if (count > 0.0) {
      const double per = per_sequence ? count * static_cast<double>(cnt[sid]) : count;
      w = static_cast<float>(1.0 / per);
    }
  }
  wrow[t] = w;
}

cudaError_t launch_weights(const uint8_t* mask, const int32_t* seq, int num_seqs, int per_sequence,
                           int64_t T, int* cnt, WsHeader* hdr, float* wrow, const int64_t* global_count,
                           cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(num_seqs) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((T + kWeightThreads - 1) / kWeightThreads);
  seq_count_kernel<<<blocks, kWeightThreads, 0, st>>>(mask, seq, T, num_seqs, cnt, &hdr->status);
  seq_total_kernel<<<1, kFinalThreads, 0, st>>>(cnt, num_seqs, per_sequence, global_count, hdr, nullptr);
  row_weight_kernel<<<blocks, kWeightThreads, 0, st>>>(mask, seq, T, num_seqs, per_sequence, cnt, hdr,
                                                      global_count, wrow);
  return cudaGetLastError();
}

cudaError_t launch_local_count(const uint8_t* mask, const int32_t* seq, int num_seqs, int per_sequence,
                               int64_t T, int* cnt, WsHeader* hdr, int64_t* count, cudaStream_t st) {
  if (T == 0) return cudaMemsetAsync(count, 0, sizeof(int64_t), st);
  cudaError_t e = cudaMemsetAsync(cnt, 0, static_cast<size_t>(num_seqs) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>((T + kWeightThreads - 1) / kWeightThreads);
  seq_count_kernel<<<blocks, kWeightThreads, 0, st>>>(mask, seq, T, num_seqs, cnt, &hdr->status);
  seq_total_kernel<<<1, kFinalThreads, 0, st>>>(cnt, num_seqs, per_sequence, nullptr, hdr, count);
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

__global__ void poison16_kernel(uint16_t* a, int64_t na, uint16_t* b, int64_t nb, const uint32_t* status) {
  if (*reinterpret_cast<const volatile uint32_t*>(status) == 0u) return;
  constexpr uint16_t kNan = 0x7FC0u;  // bf16 quiet NaN
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < na; i += stride) a[i] = kNan;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nb; i += stride) b[i] = kNan;
}

cudaError_t launch_poison16(uint16_t* a, int64_t na, uint16_t* b, int64_t nb, const uint32_t* status,
                            int sms, cudaStream_t st) {
  poison16_kernel<<<sms * 4, 256, 0, st>>>(a, na, b, nb, status);
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
