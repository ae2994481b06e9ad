// Persistent tcgen05 GEMM for sm_103a with fused epilogues.
//
// One CTA per SM, 192 threads in three roles:
//   warp 0      TMA producer: streams 128 x 64 tiles of A and BN x 64 tiles of B into a
//               STAGES-deep shared-memory ring (128-byte swizzle), one mbarrier per slot;
//   warp 1      MMA issuer: one thread issues tcgen05.mma (bf16 x bf16 -> fp32, 128 x BN
//               x 16 per instruction) into one of two TMEM accumulators and releases
//               shared-memory slots with tcgen05.commit;
//   warps 2..5  epilogue: read the finished accumulator from TMEM (each warp its own 32
//               lanes), run the fused epilogue, hand the accumulator back.
// Two accumulators (2 x BN of the 512 TMEM columns) let the epilogue of one tile overlap
// the MMAs of the next.
//
// The work is divided into units: a unit is one 128-row block of A and a contiguous range
// of n tiles.  Units are dealt round-robin to CTAs in row-block-major order, so CTAs that
// run at the same time share the same B tiles (and A blocks) in L2.  An epilogue may keep
// per-row state across the tiles of a unit (the forward's running logsumexp).
//
// Every wait is bounded (fkl_ptx.cuh): when one runs out, the kernel records
// FKL_ERR_TIMEOUT in the status word, every role stops, in-flight copies and MMAs are
// drained and TMEM is freed before the CTA exits.
#pragma once

#include <climits>
#include <cmath>

#include "fkl_ptx.cuh"

namespace fkl {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

__host__ __device__ constexpr int stages_for(int bn) { return bn == 256 ? 4 : (bn == 192 ? 5 : 6); }
__host__ __device__ constexpr size_t smem_bytes_for(int bn) {
  return static_cast<size_t>(stages_for(bn)) * (kBM * kBK * 2 + bn * kBK * 2) + 1024 + 256;
}

// Unit u -> (row block, vocabulary split).  Units are numbered in groups of group_m row
// blocks; within a group the split varies slowest, so the pairs running at the same time
// cover group_m row blocks of the same few splits and share their B tiles in L2.
__device__ __forceinline__ void unit_range(const GemmShape& g, int u, int& m_blk, int& n_begin,
                                           int& n_end, int& split) {
  const int per_group = g.group_m * g.nsplit;
  const int grp = u / per_group;
  const int r = u - grp * per_group;
  const int m0 = grp * g.group_m;
  const int rows = min(g.group_m, g.m_tiles - m0);
  split = r / rows;
  m_blk = m0 + (r - split * rows);
  n_begin = static_cast<int>(static_cast<long long>(split) * g.n_tiles / g.nsplit);
  n_end = static_cast<int>(static_cast<long long>(split + 1) * g.n_tiles / g.nsplit);
}

// Work items of the two-SM kernel: the units before g.split_from whole, then ksplit pieces of
// each later unit, a piece covering k-blocks [kb0, kb1).  slot is the piece's partial tile
// in g.kpart, or -1 for a whole unit.
__host__ __device__ __forceinline__ int num_items(const GemmShape& g) {
  return g.split_from + (g.num_units - g.split_from) * g.ksplit;
}

__device__ __forceinline__ void item_range(const GemmShape& g, int it, int& m_blk, int& n_begin, int& n_end,
                                           int& split, int& kb0, int& kb1, int& slot) {
  if (it < g.split_from) {
    unit_range(g, it, m_blk, n_begin, n_end, split);
    kb0 = 0;
    kb1 = g.k_blocks;
    slot = -1;
    return;
  }
  const int j = it - g.split_from;
  const int piece = j % g.ksplit;
  unit_range(g, g.split_from + j / g.ksplit, m_blk, n_begin, n_end, split);
  kb0 = static_cast<int>(static_cast<long long>(piece) * g.k_blocks / g.ksplit);
  kb1 = static_cast<int>(static_cast<long long>(piece + 1) * g.k_blocks / g.ksplit);
  slot = j;
}


// 256-bit global store and load (32-byte aligned addresses): one full 32-byte sector per
// thread, half the instructions of 16-byte vectors for the epilogues' row-wise output.
__device__ __forceinline__ void st_v8(void* ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                      uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d),
               "r"(e), "r"(f), "r"(g), "r"(h) : "memory");
}
__device__ __forceinline__ void ld_v8(const void* ptr, float (&x)[8]) {
  asm volatile("ld.global.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7])
               : "l"(ptr) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void pin(float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) asm volatile("" : "+f"(v[j]));
}

// ------------------------------------------------------------------ top-K cursor
// Walks one row's (id, p) pairs, sorted by id, in step with the vocabulary tiles.
struct TopkCursor {
  const int2* rowp;
  int K, kp, nid;
  float pn;

  __device__ __forceinline__ void next() {
    ++kp;
    if (kp < K) {
      const int2 e = __ldg(rowp + kp);
      nid = e.x;
      pn = __int_as_float(e.y);
    } else {
      nid = INT_MAX;
    }
  }
  // Positions the cursor on the first pair whose id is >= col.
  __device__ __forceinline__ void seek(const int2* row, int k, int col) {
    rowp = row;
    K = k;
    int lo = 0, hi = k;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(&row[mid].x) < col) lo = mid + 1; else hi = mid;
    }
    kp = lo - 1;
    next();
  }
  __device__ __forceinline__ void none() { nid = INT_MAX; }
};

// Value of v[j] for a run-time j without indexing registers dynamically.
__device__ __forceinline__ float pick(const float (&v)[32], int j) {
  float r = 0.f;
#pragma unroll
  for (int jj = 0; jj < 32; ++jj) r = (jj == j) ? v[jj] : r;
  return r;
}

// ------------------------------------------------------------------ forward epilogue
// Per row of the unit: a base-2 reference m2 and the sum l of exp2(s * log2(e)/tau - m2) over
// the vocabulary columns of the unit, and g = sum of p_k * s at the teacher ids that fall
// in the unit.  Columns >= V (zero rows that TMA filled in) are excluded.  m2 is the running
// maximum taken lazily: a 32-column chunk is first summed against m2 as it stands, and only
// when a term of it exceeds 2^32 (or m2 is not set yet, at the unit's first chunk) is the
// maximum taken again and l rescaled.  l then stays below 2^32 per chunk, far from fp32's
// range, and lse = m2 + log2(l) is the same value; the maximum's three-input max
// instructions and the rescale run only on the rare chunks that need them (in a same-process
// A/B the 32K forward took 6 % less time).
struct EpiFwd {
  using Params = FwdParams;
  const Params& p;
  int t;
  bool row_ok;
  float m2, l, g;
  TopkCursor cur;

  __device__ explicit EpiFwd(const Params& prm) : p(prm) {}

  // row0: first row of this CTA's 128 accumulator lanes.
  __device__ __forceinline__ void begin_unit(int row0, int n_begin, int /*split*/, int row) {
    t = row0 + row;
    row_ok = t < p.T;
    m2 = -INFINITY;
    l = 0.f;
    g = 0.f;
    if (row_ok) cur.seek(p.pairs + static_cast<size_t>(t) * p.K, p.K, n_begin * kVocabTile);
    else cur.none();
  }

  __device__ __forceinline__ void chunk(float (&v)[32], int col0) {
    if (col0 + 32 > p.V) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j >= p.V) v[j] = -INFINITY;
    }
    while (cur.nid < col0 + 32) {  // teacher ids inside this 32-column chunk (rare)
      const float sv = pick(v, cur.nid - col0);
      g = fmaf(cur.pn, sv, g);
      if (p.sg != nullptr) p.sg[static_cast<size_t>(t) * p.K + cur.kp] = sv;
      cur.next();
    }
    const float2 sc = make_float2(p.scale2, p.scale2);
    if (m2 != -INFINITY) {  // against the running reference as it stands
      const float2 om = make_float2(-m2, -m2);
      float2 t01 = make_float2(0.f, 0.f), t23 = make_float2(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const float2 a01 = ffma2(make_float2(v[j + 0], v[j + 1]), sc, om);
        const float2 a23 = ffma2(make_float2(v[j + 2], v[j + 3]), sc, om);
        t01 = fadd2(t01, make_float2(ex2_approx(a01.x), ex2_approx(a01.y)));
        t23 = fadd2(t23, make_float2(ex2_approx(a23.x), ex2_approx(a23.y)));
      }
      const float tsum = (t01.x + t01.y) + (t23.x + t23.y);
      if (tsum < 4294967296.f) {
        l += tsum;
        return;
      }
    }
    // the unit's first chunk, or a term above 2^32 of m2: take the maximum and rescale
    float c0 = fmax3(v[0], v[1], v[2]), c1 = fmax3(v[3], v[4], v[5]);
#pragma unroll
    for (int j = 6; j < 30; j += 4) {
      c0 = fmax3(c0, v[j], v[j + 1]);
      c1 = fmax3(c1, v[j + 2], v[j + 3]);
    }
    const float new_m = fmaxf(m2, fmax3(c0, c1, fmaxf(v[30], v[31])) * p.scale2);
    if (new_m == -INFINITY) return;  // nothing inside the vocabulary yet
    const float2 nm = make_float2(-new_m, -new_m);
    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const float2 a01 = ffma2(make_float2(v[j + 0], v[j + 1]), sc, nm);
      const float2 a23 = ffma2(make_float2(v[j + 2], v[j + 3]), sc, nm);
      s01 = fadd2(s01, make_float2(ex2_approx(a01.x), ex2_approx(a01.y)));
      s23 = fadd2(s23, make_float2(ex2_approx(a23.x), ex2_approx(a23.y)));
    }
    l = fmaf(l, ex2_approx(m2 - new_m), (s01.x + s01.y) + (s23.x + s23.y));
    m2 = new_m;
  }

  template <int BN>
  __device__ __forceinline__ void tile(uint32_t taddr, int n, int /*row*/) {
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

  __device__ __forceinline__ void end_unit(int split, int /*row*/) {
    if (!row_ok) return;
    const size_t plane = static_cast<size_t>(p.nsplit) * p.T;
    const size_t i = static_cast<size_t>(split) * p.T + t;
    p.part[i] = m2;
    p.part[plane + i] = l;
    p.part[2 * plane + i] = g;
  }
};

// ------------------------------------------------------------------ backward dS epilogue
// dS[t, v] = g tau w_t (a_t q_tv - r[t, v]) (w_t = 0 for masked rows), rounded to bf16 and
// written to the slab buffer; q_tv = exp2(s * log2(e)/tau - lse_t * log2(e)), and r is the
// pairs' second field added at their ids (for KL, a_t = 1 and r = ptilde).  The row's factor
// c_t = g tau w_t a_t is folded into the exponent: c q = sign(c) exp2(s * log2(e)/tau +
// (log2|c| - lse_t log2(e))), one packed FMA and the exponential per value instead of two
// further products; the sign is uniform across rows for KL (that of g).  The shifted
// argument rounds a little differently from the product (relative 1e-6, far below the
// bf16 output's 2^-9).  Then g tau w_t r is subtracted at the teacher ids.
struct EpiDs {
  using Params = DsParams;
  const Params& p;
  int t;
  bool row_ok, neg;
  float off, f;
  uint16_t* dst;
  TopkCursor cur;

  __device__ explicit EpiDs(const Params& prm) : p(prm) {}

  __device__ __forceinline__ void begin_unit(int row0, int n_begin, int /*split*/, int row) {
    t = row0 + row;
    row_ok = t < p.T;
    off = 0.f;
    f = 0.f;
    neg = false;
    dst = nullptr;
    cur.none();
    if (row_ok) {
      f = p.hdr->gtau * p.wrow[t];
      const float c = f * (p.arow != nullptr ? p.arow[t] : 1.f);
      neg = c < 0.f;
      off = log2f(fabsf(c)) - p.lse[t] * kLog2e;  // -inf for c = 0: the q term vanishes
      dst = p.ds + static_cast<size_t>(t) * p.ld_ds;
      cur.seek(p.pairs + static_cast<size_t>(t) * p.K, p.K, p.v0 + n_begin * kVocabTile);
    }
  }

  __device__ __forceinline__ void chunk(float (&v)[32], int cl0) {
    if (!row_ok) return;
    uint16_t* o = dst + cl0;
    if (f == 0.f) {  // a masked row (or g = 0): dS is zero
#pragma unroll
      for (int j = 0; j < 2; ++j) st_v8(o + 16 * j, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u);
      return;
    }
    const int cg0 = p.v0 + cl0;
    {
      const float2 sc = make_float2(p.scale2, p.scale2), oo = make_float2(off, off);
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const float2 x = ffma2(make_float2(v[j], v[j + 1]), sc, oo);
        v[j] = ex2_approx(x.x);
        v[j + 1] = ex2_approx(x.y);
      }
    }
    if (neg) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = -v[j];
    }
    while (cur.nid < cg0 + 32) {  // subtract g tau w_t r at the teacher ids in this chunk (rare)
      const int jt = cur.nid - cg0;
      const float d = f * cur.pn;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j == jt) v[j] -= d;
      cur.next();
    }
    if (cl0 + 32 > p.slab_w) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (cl0 + j >= p.slab_w) v[j] = 0.f;
    }
    uint32_t w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) w[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      st_v8(o + 16 * j, w[8 * j], w[8 * j + 1], w[8 * j + 2], w[8 * j + 3], w[8 * j + 4], w[8 * j + 5],
            w[8 * j + 6], w[8 * j + 7]);
  }

  template <int BN>
  __device__ __forceinline__ void tile(uint32_t taddr, int n, int /*row*/) {
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

  __device__ __forceinline__ void end_unit(int, int) {}
};

// ------------------------------------------------------------------ fp32 store epilogue
// kBf16: the tile goes to the bf16 destination (F32Params::out16); a separate instantiation,
// so that the fp32 product carries none of that path.
template <bool kBf16>
struct EpiF32T {
  using Params = F32Params;
  const Params& p;
  bool row_ok;
  bool part;  // the tile is one K piece, stored whole to a partial tile (row stride BN)
  float* rowp;
  uint16_t* rowp16;

  __device__ explicit EpiF32T(const Params& prm) : p(prm) {}

  __device__ __forceinline__ void begin_unit(int row0, int, int, int row) {
    const int r = row0 + row;
    row_ok = r < p.M;
    part = false;
    const size_t rr = static_cast<size_t>(row_ok ? r : 0);
    rowp = p.out != nullptr ? p.out + rr * p.ldo : nullptr;
    rowp16 = p.out16 != nullptr ? p.out16 + rr * p.ldo16 : nullptr;
  }

  // bf16 destination: adds the fp32 sum so far when accumulating, rounds to nearest even.
  __device__ __forceinline__ void store16(float (&v)[32], int col0) {
    const bool full = col0 + 32 <= p.N;
    if (p.accumulate) {
      const float* src = rowp + col0;
      if (p.vec_ok && full) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float y[8];
          ld_v8(src + 8 * j, y);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[8 * j + i] += y[i];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col0 + j < p.N) v[j] += src[j];
      }
    }
    uint16_t* o = rowp16 + col0;
    if (p.vec16_ok && full) {
      uint4* o4 = reinterpret_cast<uint4*>(o);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        o4[j] = make_uint4(pack_bf16x2(v[8 * j + 0], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                           pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.N) o[j] = static_cast<uint16_t>(pack_bf16x2(v[j], 0.f) & 0xFFFFu);
    }
  }

  // A K piece: this thread's row of the partial tile at `tile` (ld floats per row).
  __device__ __forceinline__ void begin_part(float* tile, int ld, int row0, int row_in_tile, int row) {
    row_ok = row0 + row < p.M;
    part = true;
    rowp = tile + static_cast<size_t>(row_in_tile) * ld;
  }

  template <int BN>
  __device__ __forceinline__ void tile(uint32_t taddr, int n, int) {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = n * BN + c * 32;
      if (col0 >= p.N) break;  // same for the whole warp
      float v[32];
      tmem_ld32(taddr + c * 32, v);
      tmem_ld_wait(v);
      if (!row_ok) continue;
      if constexpr (kBf16) {
        if (!part) {
          store16(v, col0);
          continue;
        }
      }
      float* o = part ? rowp + c * 32 : rowp + col0;
      if (part || (p.vec_ok && col0 + 32 <= p.N)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = v[8 * j + i];
          if (p.accumulate && !part) {
            float y[8];
            ld_v8(o + 8 * j, y);
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] += y[i];
          }
          st_v8(o + 8 * j, __float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]), __float_as_uint(x[3]),
                __float_as_uint(x[4]), __float_as_uint(x[5]), __float_as_uint(x[6]), __float_as_uint(x[7]));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (col0 + j < p.N) o[j] = p.accumulate ? o[j] + v[j] : v[j];
        }
      }
    }
  }

  __device__ __forceinline__ void end_unit(int, int) {}
};
using EpiF32 = EpiF32T<false>;
using EpiF32Bf16 = EpiF32T<true>;

// ------------------------------------------------------------------ the kernel
// Shared-memory layout of the one-SM kernel for a B tile of BN rows.
template <int BN>
struct SmLayout {
  static constexpr int STAGES = stages_for(BN);
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;  // 16 KB
  static constexpr uint32_t B_BYTES = BN * kBK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t BOX_BYTES = 64 * kBK * 2;  // one 64 x 64 MN-major box, 8 KB
};

// What every role of a CTA needs: the shared-memory ring and barriers, the TMEM
// accumulators and the bounded-wait control.
struct SmCtx {
  uint32_t stage0, full0, empty0, tfull0, tempty0, drain;
  uint32_t tmem_base;
  WaitCtl ctl;
};

// TMA producer (lane 0 of warp 0).
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ void sm_producer(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmShape& g,
                                            const SmCtx& c) {
  using L = SmLayout<BN>;
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_par = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < g.num_units; u += gridDim.x) {
    int m_blk, nb, ne, split;
    unit_range(g, u, m_blk, nb, ne, split);
    for (int n = nb; ok && n < ne; ++n) {
      for (int kb = 0; kb < g.k_blocks; ++kb) {
        if (!mbar_wait(c.empty0 + 8 * stage, phase ^ 1u, c.ctl)) { ok = false; break; }
        const uint32_t fb = c.full0 + 8 * stage;
        const uint32_t sa = c.stage0 + stage * L::STAGE_BYTES;
        const uint32_t sb = sa + L::A_BYTES;
        const int k0 = kb * kBK;
        mbar_arrive_expect_tx(fb, L::STAGE_BYTES);
        if (!A_MN) {
          tma_load_2d(sa, tmA, fb, k0, m_blk * kBM);
        } else if (g.a_box3d) {
          tma_load_3d(sa, tmA, fb, 0, k0, m_blk * (kBM / 64));
        } else {
          tma_load_2d(sa, tmA, fb, m_blk * kBM, k0);
          tma_load_2d(sa + L::BOX_BYTES, tmA, fb, m_blk * kBM + 64, k0);
        }
        if (!B_MN) {
          tma_load_2d(sb, tmB, fb, k0, n * BN);
        } else if (g.b_box3d) {
          tma_load_3d(sb, tmB, fb, 0, k0, n * (BN / 64));
        } else {
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + j * L::BOX_BYTES, tmB, fb, n * BN + j * 64, k0);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == L::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
  }
  // Every copy this thread started must land before the CTA may exit.
  for (int s = 0; s < L::STAGES; ++s)
    if ((issued >> s) & 1u) mbar_wait_drain(c.full0 + 8 * s, (issued_par >> s) & 1u, g.limit_ns);
}

// MMA issuer (lane 0 of warp 1): 128 x BN x 16 MMAs into one of two TMEM accumulators.
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ void sm_mma(const GemmShape& g, const SmCtx& c) {
  using L = SmLayout<BN>;
  constexpr uint32_t IDESC = instr_desc_bf16(kBM, BN, A_MN, B_MN);
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < g.num_units; u += gridDim.x) {
    int m_blk, nb, ne, split;
    unit_range(g, u, m_blk, nb, ne, split);
    for (int n = nb; ok && n < ne; ++n) {
      if (!mbar_wait(c.tempty0 + 8 * acc, acc_phase ^ 1u, c.ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = c.tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = 0; kb < g.k_blocks; ++kb) {
        if (!mbar_wait(c.full0 + 8 * stage, phase, c.ctl)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = c.stage0 + stage * L::STAGE_BYTES;
        const uint32_t sb = sa + L::A_BYTES;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k) {
          // K-major: the 16-element step moves 32 bytes along the swizzled 128-byte row.
          // MN-major: it moves 16 rows of 128 bytes; 64-wide MN blocks are 8 KB apart.
          const uint64_t ad = A_MN ? smem_desc_sw128(sa + k * 2048, L::BOX_BYTES, 1024)
                                   : smem_desc_sw128(sa + k * 32, 16, 1024);
          const uint64_t bd = B_MN ? smem_desc_sw128(sb + k * 2048, L::BOX_BYTES, 1024)
                                   : smem_desc_sw128(sb + k * 32, 16, 1024);
          tc_mma_bf16(d_tmem, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
        }
        tc_commit(c.empty0 + 8 * stage);  // slot is free once these MMAs have read it
        if (++stage == L::STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      tc_commit(c.tfull0 + 8 * acc);  // accumulator complete
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }
  // Every MMA issued must finish before TMEM is released.
  tc_commit(c.drain);
  mbar_wait_drain(c.drain, 0u, g.limit_ns);
}

// Epilogue (warps 2-5): each warp reads its 32 TMEM lanes of a finished tile and runs the
// fused epilogue.
template <int BN, class Epi>
__device__ __forceinline__ void sm_epilogue(const GemmShape& g, const typename Epi::Params& ep, const SmCtx& c,
                                            int warp, int lane) {
  const int row = (warp & 3) * 32 + lane;  // TMEM lane = row of the 128-row tile
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  Epi epi(ep);
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  for (int u = blockIdx.x; ok && u < g.num_units; u += gridDim.x) {
    int m_blk, nb, ne, split;
    unit_range(g, u, m_blk, nb, ne, split);
    epi.begin_unit(m_blk * kBM, nb, split, row);
    for (int n = nb; n < ne; ++n) {
      const bool got = mbar_wait(c.tfull0 + 8 * acc, acc_phase, c.ctl);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      epi.template tile<BN>(c.tmem_base + lane_base + static_cast<uint32_t>(acc * BN), n, row);
      tc_fence_before();
      mbar_arrive(c.tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (ok) epi.end_unit(split, row);
  }
}

template <int BN, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmShape g, const __grid_constant__ typename Epi::Params ep) {
  using L = SmLayout<BN>;
  static_assert(2 * BN <= static_cast<int>(kTmemCols), "two accumulators must fit in TMEM");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B is loaded in 64-column boxes");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::STAGES * L::STAGE_BYTES);
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 2 * L::STAGES + 5);  // [0] TMEM base, [1] abort

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = full0 + 8 * L::STAGES;
  const uint32_t tfull0 = empty0 + 8 * L::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 4 * 32);
    }
    mbar_init(drain, 1);
    misc[1] = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const WaitCtl ctl{reinterpret_cast<volatile uint32_t*>(&misc[1]), g.status, g.limit_ns};

  const SmCtx c{stage0, full0, empty0, tfull0, tempty0, drain, tmem_base, ctl};
  if (warp == 0) {
    if (lane == 0) sm_producer<BN, A_MN, B_MN>(&tmA, &tmB, g, c);
  } else if (warp == 1) {
    if (lane == 0) sm_mma<BN, A_MN, B_MN>(g, c);
  } else {
    sm_epilogue<BN, Epi>(g, ep, c, warp, lane);
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Host-side launch state of one kernel instantiation, per device: whether its dynamic
// shared-memory limit was raised, and how many clusters of it fit at once.  It lives in a
// function with internal linkage, so every copy of this library (and every translation
// unit) keeps its own: a static local of an externally visible template would be merged
// across two copies of the library loaded into one process, and the second copy would then
// skip raising the limit for its own kernels.
template <class Key>
struct LaunchState {
  bool limit_set[128];
  int clusters[128];
};
namespace {
template <class Key>
LaunchState<Key>& launch_state() {
  static LaunchState<Key> s = {};
  return s;
}
}  // namespace
template <int Kind, int BN, bool A_MN, bool B_MN, class Epi>
struct KernelKey {};

// Raises the kernel's dynamic shared-memory limit once per device (`done`: the launch state
// of this instantiation), so that later launches, including launches recorded into a CUDA
// graph, make no attribute call.
template <class Kern>
cudaError_t smem_limit_once(Kern kern, size_t smem, bool (&done)[128]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < 128;
  if (slot && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess && slot) done[dev] = true;
  return e;
}

template <int BN, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm_t(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                          const typename Epi::Params& ep, int grid, cudaStream_t st) {
  constexpr size_t SMEM = smem_bytes_for(BN);
  auto kern = gemm_kernel<BN, A_MN, B_MN, Epi>;
  cudaError_t e = smem_limit_once(kern, SMEM, launch_state<KernelKey<1, BN, A_MN, B_MN, Epi>>().limit_set);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, SMEM, st>>>(a, b, g, ep);
  return cudaGetLastError();
}

}  // namespace fkl
