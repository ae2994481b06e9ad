// Two-SM variant of the persistent tcgen05 GEMM (cta_group::2): a cluster of two CTAs on
// neighbouring SMs computes 256 x BN tiles.  Each CTA loads its own 128 rows of A and its
// own half (BN/2 rows) of B into its shared memory; the even CTA issues 256 x BN x 16
// tcgen05.mma instructions that read both CTAs' shared memory and write each CTA's 128
// accumulator rows into that CTA's TMEM.  Per SM this halves the B-operand traffic of the
// one-SM kernel (fkl_gemm.cuh): 32 KB per 64-deep k-block instead of 48 KB for BN = 256.
//
// Roles per CTA (192 threads), as in the one-SM kernel, with these hand-offs:
//   warp 0      TMA producer (both CTAs): loads into its own stage slot; the completion of
//               both CTAs' loads is counted on the even CTA's `full` barrier (the even
//               producer posts the expected bytes of the pair, 2 x STAGE_BYTES);
//   warp 1      even CTA: MMA issuer; commits slot release to `empty` and tile completion
//               to `tfull` of both CTAs (multicast commit); idle in the odd CTA;
//   warps 2..5  epilogue (both CTAs) on its own 128 TMEM lanes; hands the accumulator
//               back by arriving on the even CTA's `tempty` (8 arrivals: 4 warps x 2 CTAs).
// All three roles walk the same sequence of work items (item_range): whole units, then, for
// the fp32 products, the K pieces of the last wave's units (GemmShape::split_from), whose
// partial tiles a fixup kernel adds up afterwards.  Items are dealt round-robin to the pairs,
// or, for long launches (GemmShape::sched), drawn one at a time from a global counter by
// the even CTA's producer, which hands each to the pair's other roles through a small ring
// in shared memory.  Pairs run at slightly different speeds (1-2 % from SM to SM); with a
// fixed deal the difference accumulates over a long launch, the pairs that share a W tile
// drift apart by tens of tiles and the L2 re-reads W from DRAM, while drawing items keeps
// the pairs on neighbouring units and balances the last wave.
// Every wait is bounded as in the one-SM kernel; teardown drains copies and MMAs, meets
// the other CTA at a cluster barrier and frees TMEM of both CTAs together.
#pragma once

#include <type_traits>

#include "fkl_gemm.cuh"

namespace fkl {

constexpr int kBM2 = 256;  // rows per CTA pair

__host__ __device__ constexpr int stages2_for(int bn) { return bn == 256 ? 7 : 8; }
// An MN-major B half that is not a whole number of 64-element (128-byte) rows uses the
// 64-byte swizzle: 32-element atoms (a 192-wide tile: 96-wide halves, three atoms).
__host__ __device__ constexpr bool b_sw64_for(int bn, bool b_mn) { return b_mn && (bn / 2) % 64 != 0; }
__host__ __device__ constexpr size_t smem2_bytes_for(int bn) {
  // the operand stages, 1024 bytes of alignment slack, 512 for the barriers and other words
  return static_cast<size_t>(stages2_for(bn)) * (kBM * kBK * 2 + (bn / 2) * kBK * 2) + 1024 + 512;
}
static_assert((2 * 8 + 5 + 2 * 4) * 8 + (2 + 4) * 4 <= 512, "barriers and words fit in their 512 bytes");

// Shared-memory layout of the two-SM kernel for a B tile of BN rows (BN / 2 per CTA).
template <int BN, bool B_MN>
struct PairLayout {
  static constexpr int STAGES = stages2_for(BN);
  static constexpr int BNH = BN / 2;                   // rows of B held by each CTA
  static constexpr uint32_t A_BYTES = kBM * kBK * 2;   // 16 KB
  static constexpr uint32_t B_BYTES = BNH * kBK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t BOX_BYTES = 64 * kBK * 2;
  static constexpr bool B_SW64 = b_sw64_for(BN, B_MN);
  static constexpr uint32_t BOX64_BYTES = 32 * kBK * 2;  // one 32 x 64 MN-major box (64-byte swizzle), 4 KB
};

// What every role of one CTA of a pair needs: its place in the pair and the grid, the
// shared-memory ring and barriers, the TMEM accumulators and the bounded-wait control.
struct PairCtx {
  uint32_t rank;
  bool even;
  int cluster, nclusters;
  uint32_t stage0, full0, empty0, tfull0, tempty0, drain;
  uint32_t sfull0, sempty0, ring0;  // work-item ring (dynamic scheduling)
  uint32_t tmem_base;
  WaitCtl ctl;
};

// Work-item ring of a dynamically scheduled launch: slots in each CTA's shared memory, a
// `sfull` barrier per slot in each CTA (one arrival: the even producer's) and a `sempty`
// barrier per slot in the even CTA (one arrival per consumer: the even MMA thread, the odd
// producer and the four epilogue warps of each CTA).
constexpr int kSchedSlots = 4;
constexpr uint32_t kSchedConsumers = 10;

// The sequence of work items of one role: `it` is the current item (>= num_items: done).
struct ItemSeq {
  int it;
  int slot;
  uint32_t parity;
  __device__ explicit ItemSeq(const PairCtx& c) : it(c.cluster), slot(0), parity(0u) {}
  __device__ __forceinline__ void advance() {
    if (++slot == kSchedSlots) {
      slot = 0;
      parity ^= 1u;
    }
  }
};

// The even CTA's producer moves to its next item: the next round-robin one, or one drawn from
// the counter and published to both CTAs' rings.  False when a wait ran out.
__device__ __forceinline__ bool item_publish(const GemmShape& g, const PairCtx& c, ItemSeq& q) {
  if (g.sched == nullptr) {
    q.it += c.nclusters;
    return true;
  }
  int v = c.nclusters + (atomicAdd(g.sched, 1) - g.sched_base);
  // A counter behind this launch's base means an earlier launch of the call stopped early
  // (its wait ran out and the status word already holds the error): take no further item
  // rather than one of the first, fixed ones.
  if (v < c.nclusters) v = num_items(g);
  if (!mbar_wait_acquire_cluster(c.sempty0 + 8 * q.slot, q.parity ^ 1u, c.ctl)) return false;
  const uint32_t r = c.ring0 + 4 * static_cast<uint32_t>(q.slot);
  const uint32_t f = c.sfull0 + 8 * static_cast<uint32_t>(q.slot);
  st_shared_cluster_u32(map_to_rank(r, 0), static_cast<uint32_t>(v));
  st_shared_cluster_u32(map_to_rank(r, 1), static_cast<uint32_t>(v));
  mbar_arrive_release_cluster(map_to_rank(f, 0));
  mbar_arrive_release_cluster(map_to_rank(f, 1));
  q.advance();
  q.it = v;
  return true;
}

// Every other role moves to its next item.  For a published item the caller then releases
// the slot with item_release (once per consuming thread or warp, after it has read the
// item); `slot` receives the slot to release, -1 when there is none.  False when a wait ran out.
__device__ __forceinline__ bool item_take(const GemmShape& g, const PairCtx& c, ItemSeq& q, int& slot) {
  slot = -1;
  if (g.sched == nullptr) {
    q.it += c.nclusters;
    return true;
  }
  if (!mbar_wait_acquire_cluster(c.sfull0 + 8 * q.slot, q.parity, c.ctl)) return false;
  q.it = static_cast<int>(ld_shared_u32(c.ring0 + 4 * static_cast<uint32_t>(q.slot)));
  slot = q.slot;
  q.advance();
  return true;
}
__device__ __forceinline__ void item_release(const PairCtx& c, int slot) {
  if (slot >= 0) mbar_arrive_release_cluster(map_to_rank(c.sempty0 + 8 * static_cast<uint32_t>(slot), 0));
}

// TMA producer (lane 0 of warp 0, both CTAs): loads this CTA's A rows and half of B into the
// ring; the even CTA's `full` barrier counts the bytes of both CTAs.
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ void pair_producer(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmShape& g,
                                              const PairCtx& c) {
  using L = PairLayout<BN, B_MN>;
  const uint32_t full0_even = map_to_rank(c.full0, 0);  // the pair's `full` barriers
  int stage = 0;
  uint32_t phase = 0, issued = 0, issued_par = 0;
  bool ok = true;
  const int items = num_items(g);
  for (ItemSeq q(c); ok && q.it < items;) {
    int m_blk, nb, ne, split, kb0, kb1, slot;
    item_range(g, q.it, m_blk, nb, ne, split, kb0, kb1, slot);
    const int a_row = m_blk * kBM2 + static_cast<int>(c.rank) * kBM;
    for (int n = nb; ok && n < ne; ++n) {
      const int b_row = n * BN + static_cast<int>(c.rank) * L::BNH;
      for (int kb = kb0; kb < kb1; ++kb) {
        // the slot is released by the even CTA's tensor core (multicast commit)
        if (!mbar_wait_cluster(c.empty0 + 8 * stage, phase ^ 1u, c.ctl)) { ok = false; break; }
        const uint32_t fb = full0_even + 8 * stage;
        const uint32_t sa = c.stage0 + stage * L::STAGE_BYTES;
        const uint32_t sb = sa + L::A_BYTES;
        const int k0 = kb * kBK;
        if (c.even) mbar_arrive_expect_tx(c.full0 + 8 * stage, 2 * L::STAGE_BYTES);
        if (!A_MN) {
          tma_load_2d_pair(sa, tmA, fb, k0, a_row);
        } else if (g.a_box3d) {
          tma_load_3d_pair(sa, tmA, fb, 0, k0, a_row / 64);
        } else {
          tma_load_2d_pair(sa, tmA, fb, a_row, k0);
          tma_load_2d_pair(sa + L::BOX_BYTES, tmA, fb, a_row + 64, k0);
        }
        if (!B_MN) {
          tma_load_2d_pair(sb, tmB, fb, k0, b_row);
        } else if (L::B_SW64) {
          if (g.b_box3d) {
            tma_load_3d_pair(sb, tmB, fb, 0, k0, b_row / 32);
          } else {
#pragma unroll
            for (int j = 0; j < L::BNH / 32; ++j) tma_load_2d_pair(sb + j * L::BOX64_BYTES, tmB, fb, b_row + j * 32, k0);
          }
        } else if (g.b_box3d) {
          tma_load_3d_pair(sb, tmB, fb, 0, k0, b_row / 64);
        } else {
#pragma unroll
          for (int j = 0; j < L::BNH / 64; ++j) tma_load_2d_pair(sb + j * L::BOX_BYTES, tmB, fb, b_row + j * 64, k0);
        }
        issued |= 1u << stage;
        issued_par = (issued_par & ~(1u << stage)) | (phase << stage);
        if (++stage == L::STAGES) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) break;
    if (c.even) {
      ok = item_publish(g, c, q);
    } else {
      int rel;
      ok = item_take(g, c, q, rel);
      item_release(c, rel);
    }
  }
  // The even CTA drains the pair's copies (its `full` phases count both CTAs' bytes).
  // The odd CTA's copies are covered by those phases; on the abort path its last copy
  // was issued before a wait that ran for the full time limit.
  if (c.even)
    for (int s = 0; s < L::STAGES; ++s)
      if ((issued >> s) & 1u) mbar_wait_drain(c.full0 + 8 * s, (issued_par >> s) & 1u, g.limit_ns);
}

// MMA issuer (lane 0 of warp 1, even CTA): 256 x BN x 16 MMAs into one of two TMEM
// accumulators; commits free ring slots and announce finished tiles to both CTAs.
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ void pair_mma(const GemmShape& g, const PairCtx& c) {
  using L = PairLayout<BN, B_MN>;
  constexpr uint32_t IDESC = instr_desc_bf16(kBM2, BN, A_MN, B_MN);
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool ok = true;
  const int items = num_items(g);
  // Shared-memory descriptors of stage 0 at k-slice 0, built once.  A descriptor holds the
  // start address / 16 in its low 14 bits, and every operand address stays below 256 KB,
  // so the descriptor of another stage or k-slice is this one plus that offset / 16 (the
  // swizzled layouts put 16-deep slices 32 bytes apart in a K-major tile, 2048 bytes apart
  // in a 128-byte-swizzled MN-major one and 1024 in a 64-byte-swizzled MN-major B).  Fewer
  // instructions on the issuing thread made the forward 2 % faster at 32K.
  const uint32_t sb0 = c.stage0 + L::A_BYTES;
  const uint64_t a_desc0 = A_MN ? smem_desc_sw128(c.stage0, L::BOX_BYTES, 1024) : smem_desc_sw128(c.stage0, 16, 1024);
  const uint64_t b_desc0 = !B_MN ? smem_desc_sw128(sb0, 16, 1024)
                           : L::B_SW64 ? smem_desc(sb0, L::BOX64_BYTES, 512, 4u)
                                    : smem_desc_sw128(sb0, L::BOX_BYTES, 1024);
  constexpr uint64_t kStageStep = L::STAGE_BYTES >> 4;
  constexpr uint64_t kAStep = (A_MN ? 2048u : 32u) >> 4;
  constexpr uint64_t kBStep = (!B_MN ? 32u : L::B_SW64 ? 1024u : 2048u) >> 4;
  uint64_t a_stage = a_desc0, b_stage = b_desc0;
  for (ItemSeq q(c); ok && q.it < items;) {
    int m_blk, nb, ne, split, kb0, kb1, slot;
    item_range(g, q.it, m_blk, nb, ne, split, kb0, kb1, slot);
    for (int n = nb; ok && n < ne; ++n) {
      if (!mbar_wait_cluster(c.tempty0 + 8 * acc, acc_phase ^ 1u, c.ctl)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_tmem = c.tmem_base + static_cast<uint32_t>(acc * BN);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait_cluster(c.full0 + 8 * stage, phase, c.ctl)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          tc_mma_bf16_pair(d_tmem, a_stage + k * kAStep, b_stage + k * kBStep, IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
        tc_commit_pair_mc(c.empty0 + 8 * stage, 0x3);  // frees the slot in both CTAs
        if (++stage == L::STAGES) {
          stage = 0;
          phase ^= 1u;
          a_stage = a_desc0;
          b_stage = b_desc0;
        } else {
          a_stage += kStageStep;
          b_stage += kStageStep;
        }
      }
      if (!ok) break;
      tc_commit_pair_mc(c.tfull0 + 8 * acc, 0x3);  // both halves of the tile are complete
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) break;
    int rel;
    ok = item_take(g, c, q, rel);
    item_release(c, rel);
  }
  tc_commit_pair(c.drain);
  mbar_wait_drain(c.drain, 0u, g.limit_ns);
}

// Epilogue (warps 2-5, both CTAs): each warp reads its 32 TMEM lanes of a finished tile,
// runs the fused epilogue and hands the accumulator back to the even CTA.
template <int BN, class Epi>
__device__ __forceinline__ void pair_epilogue(const GemmShape& g, const typename Epi::Params& ep, const PairCtx& c,
                                              int warp, int lane) {
  const int row = (warp & 3) * 32 + lane;
  const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t remote_tempty0 = map_to_rank(c.tempty0, 0);
  Epi epi(ep);
  int acc = 0;
  uint32_t acc_phase = 0;
  bool ok = true;
  const int items = num_items(g);
  for (ItemSeq q(c); ok && q.it < items;) {
    int m_blk, nb, ne, split, kb0, kb1, slot;
    item_range(g, q.it, m_blk, nb, ne, split, kb0, kb1, slot);
    const int row0 = m_blk * kBM2 + static_cast<int>(c.rank) * kBM;
    if constexpr (std::is_same<Epi, EpiF32>::value || std::is_same<Epi, EpiF32Bf16>::value) {
      if (slot >= 0)
        epi.begin_part(g.kpart + static_cast<size_t>(slot) * (kBM2 * BN), BN, row0,
                       static_cast<int>(c.rank) * kBM + row, row);
      else
        epi.begin_unit(row0, nb, split, row);
    } else {
      epi.begin_unit(row0, nb, split, row);
    }
    for (int n = nb; n < ne; ++n) {
      const bool got = mbar_wait_cluster(c.tfull0 + 8 * acc, acc_phase, c.ctl);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      epi.template tile<BN>(c.tmem_base + lane_base + static_cast<uint32_t>(acc * BN), n, row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(remote_tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok) break;
    epi.end_unit(split, row);
    int rel;
    ok = __all_sync(0xffffffffu, item_take(g, c, q, rel));
    __syncwarp();
    if (lane == 0) item_release(c, rel);
  }
}

template <int BN, bool A_MN, bool B_MN, class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const GemmShape g, const __grid_constant__ typename Epi::Params ep) {
  using L = PairLayout<BN, B_MN>;
  static_assert(BN == 256 || BN == 192 || BN == 128, "two-SM tiles are 256 x {256, 192, 128}");
  static_assert(!L::B_SW64 || (BN / 2) % 32 == 0, "64-byte swizzle halves are whole 32-wide atoms");
  static_assert(2 * BN <= static_cast<int>(kTmemCols), "two accumulators must fit in TMEM");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::STAGES * L::STAGE_BYTES);
  // [0] TMEM base, [1] abort, [2, 2 + kSchedSlots) work-item ring
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + 2 * L::STAGES + 5 + 2 * kSchedSlots);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool even = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = full0 + 8 * L::STAGES;
  const uint32_t tfull0 = empty0 + 8 * L::STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t sfull0 = drain + 8;
  const uint32_t sempty0 = sfull0 + 8 * kSchedSlots;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull0 + 8 * b, 1);
      mbar_init(tempty0 + 8 * b, 2 * 4);
    }
    mbar_init(drain, 1);
    for (int k = 0; k < kSchedSlots; ++k) {
      mbar_init(sfull0 + 8 * k, 1);
      mbar_init(sempty0 + 8 * k, kSchedConsumers);
    }
    misc[1] = 0u;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(&misc[0]), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = misc[0];
  const WaitCtl ctl{reinterpret_cast<volatile uint32_t*>(&misc[1]), g.status, g.limit_ns};

  const PairCtx c{rank,   even,   cluster, nclusters,          stage0,   full0,    empty0, tfull0,
                  tempty0, drain, sfull0,  sempty0, smem_addr(&misc[2]), tmem_base, ctl};
  if (warp == 0) {
    if (lane == 0) pair_producer<BN, A_MN, B_MN>(&tmA, &tmB, g, c);
  } else if (warp == 1) {
    if (lane == 0 && even) pair_mma<BN, A_MN, B_MN>(g, c);
  } else {
    pair_epilogue<BN, Epi>(g, ep, c, warp, lane);
  }

  __syncthreads();
  tc_fence_before();
  cluster_sync();  // no arrival or commit toward either CTA is still in flight
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Clusters of one kernel instantiation that fit on the device at once, cached per device in
// `cached` (one array per instantiation: the occupancy depends on its shared memory).
template <class Kern>
int max_pair_clusters(Kern kern, size_t smem, int sms, int (&cached)[128]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  if (n > sms / 2) n = sms / 2;
  cached[dev] = n;
  return n;
}

template <int BN, bool A_MN, bool B_MN, class Epi>
cudaError_t launch_gemm2_t(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                           const typename Epi::Params& ep, int sms, cudaStream_t st) {
  constexpr size_t SMEM = smem2_bytes_for(BN);
  auto kern = gemm2_kernel<BN, A_MN, B_MN, Epi>;
  LaunchState<KernelKey<2, BN, A_MN, B_MN, Epi>>& state = launch_state<KernelKey<2, BN, A_MN, B_MN, Epi>>();
  cudaError_t e = smem_limit_once(kern, SMEM, state.limit_set);
  if (e != cudaSuccess) return e;
  const int clusters = max_pair_clusters(kern, SMEM, sms, state.clusters);
  const int items = num_items(g);
  const int n = items < clusters ? items : clusters;
  kern<<<2 * n, kThreads, SMEM, st>>>(a, b, g, ep);
  return cudaGetLastError();
}

}  // namespace fkl
