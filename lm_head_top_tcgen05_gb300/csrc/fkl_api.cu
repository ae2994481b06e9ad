// Host side of the C ABI (include/fkl.h, include/fkl_testing.h; the teacher cache producer is
// in fkl_topk.cu, the allocation-free forward in fkl_noalloc.cu): argument checks, the
// workspace plan, tensor-map encoding, the tile schedule and the launch sequences of the
// forward and backward passes.  All work is enqueued on the caller's stream; nothing here
// allocates device memory or synchronises, except fkl_read_status.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fkl.h"
#include "../../include/fkl_testing.h"
#include "fkl_internal.h"

namespace fkl {

static thread_local std::string g_last_error;

static fkl_status fail(fkl_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

void set_last_error_message(const char* msg) { g_last_error = msg; }

int check_device_memory(const NamedPtr* ptrs, int n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(FKL_ERR_CUDA, "cudaGetDevice failed");
  for (int i = 0; i < n; ++i) {
    if (ptrs[i].p == nullptr) continue;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptrs[i].p) != cudaSuccess) {
      cudaGetLastError();
      return fail(FKL_ERR_INVALID_ARG, "%s is not CUDA memory", ptrs[i].name);
    }
    const bool ok = (a.type == cudaMemoryTypeDevice && a.device == dev) || a.type == cudaMemoryTypeManaged;
    if (!ok) return fail(FKL_ERR_INVALID_ARG, "%s is not device memory of the current device", ptrs[i].name);
  }
  return FKL_OK;
}

static fkl_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FKL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
static inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool make_plan(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk, Plan* p, bool bf16_grads,
               int max_splits) {
  if (T < 0 || T >= (int64_t{1} << 31)) return false;
  if (d < 8 || d % 8 != 0 || d >= (int64_t{1} << 20)) return false;
  if (V < 1 || V > (int64_t{1} << 30)) return false;
  if (K < 1 || K > 1024) return false;
  if (chunk < 1) return false;
  p->T = T; p->d = d; p->V = V; p->K = K; p->chunk = chunk;
  const int64_t vpad = cdiv(V, kVocabTile) * kVocabTile;
  if (T == 0) {
    p->Ct = 0;
    p->nt = 0;
    p->Vc = kVocabTile;
    p->Vmax = kVocabTile;
    p->nslabs = 0;
  } else {
    // The backward walks blocks of Ct tokens x Vc vocabulary columns; the dS buffer of one
    // block holds at most chunk * V values (Vc whole 256-column tiles, at least one, evened
    // out over the slabs).  dH is rewritten once per vocabulary slab and dW once per token
    // block; full-height slabs (Ct = T) write dW once, and lower blocks are taken only when
    // they cut that read-modify-write traffic by a quarter or more (long sequences).
    const int64_t budget = (chunk < T ? chunk : T) * V;
    auto width = [&](int64_t ct) {
      int64_t vc = budget / ct;
      vc = (vc / kVocabTile) * kVocabTile;
      if (vc < kVocabTile) vc = kVocabTile;
      if (vc > vpad) vc = vpad;
      const int64_t ns = cdiv(V, vc);
      const int64_t even = cdiv(cdiv(V, ns), kVocabTile) * kVocabTile;
      return even < vc ? even : vc;
    };
    auto rmw = [&](int64_t nt, int64_t ns) {  // bytes of dH and dW traffic
      return static_cast<double>(2 * ns - 1) * T * d * 4 + static_cast<double>(2 * nt - 1) * V * d * 4;
    };
    int64_t best_ct = T, best_vc = width(T);
    const double full = rmw(1, cdiv(V, best_vc));
    double best = full;
    for (int64_t n = 2; n <= kMaxTokenBlocks; ++n) {
      const int64_t ct = cdiv(cdiv(T, n), kVocabTile) * kVocabTile;
      if (ct >= T) continue;
      const int64_t vc = width(ct);
      const double c = rmw(cdiv(T, ct), cdiv(V, vc));
      if (c < best) { best = c; best_ct = ct; best_vc = vc; }
    }
    if (best > 0.75 * full) { best_ct = T; best_vc = width(T); }
    p->Ct = best_ct;
    p->nt = cdiv(T, best_ct);
    p->Vc = best_vc;
    p->nslabs = cdiv(V, p->Vc);
    int64_t vmax = (budget / best_ct / kVocabTile) * kVocabTile;
    if (vmax > vpad) vmax = vpad;
    p->Vmax = vmax > best_vc ? vmax : best_vc;
  }
  p->nb = cdiv(T, 256);
  size_t off = 256;  // header
  p->off_pairs = off; off = align_up(off + static_cast<size_t>(T) * K * 8, 256);
  p->off_crow = off;  off = align_up(off + static_cast<size_t>(T) * 4, 256);
  p->off_wrow = off;  off = align_up(off + static_cast<size_t>(T) * 4, 256);
  p->off_scnt = off;  off = align_up(off + static_cast<size_t>(T > 0 ? T : 1) * 4, 256);
  p->off_part = off;  off = align_up(off + static_cast<size_t>(T) * 3 * max_splits * 4, 256);
  const size_t nbb = static_cast<size_t>(p->nb > 0 ? p->nb : 1);
  p->off_bsum = off;  off = align_up(off + nbb * 8, 256);
  p->off_bcnt = off;  off = align_up(off + nbb * 4, 256);
  p->off_ds = off;    off = align_up(off + static_cast<size_t>(p->Ct) * p->Vmax * 2, 256);
  p->off_slot = off;  off = align_up(off + static_cast<size_t>(T) * K * 4, 256);
  p->off_sg = off;    off = align_up(off + static_cast<size_t>(T) * K * 4, 256);
  p->off_arow = off;  off = align_up(off + static_cast<size_t>(T) * 4, 256);
  p->off_kpart = off;
  if (T > 0) off = align_up(off + static_cast<size_t>(kKsplitSlots) * 256 * 256 * 4, 256);
  // bf16 gradients: with several token blocks, walk the slabs in the outer loop when its
  // fp32 sums (all of dH, one slab of dW) are smaller than the other order's (one block of
  // dH, all of dW); the summation orders are the same either way
  p->slab_outer = false;
  size_t hsum = 0, wsum = 0;
  if (bf16_grads && T > 0) {
    hsum = static_cast<size_t>(p->Ct) * d * 4;
    if (p->nt > 1) {
      wsum = static_cast<size_t>(V) * d * 4;
      const size_t h2 = static_cast<size_t>(T) * d * 4, w2 = static_cast<size_t>(p->Vmax) * d * 4;
      if (h2 + w2 < hsum + wsum) {
        p->slab_outer = true;
        hsum = h2;
        wsum = w2;
      }
    }
  }
  p->off_hsum = off;
  if (hsum) off = align_up(off + hsum, 256);
  p->off_wsum = off;
  if (wsum) off = align_up(off + wsum, 256);
  p->total = off;
  return true;
}

// Critical path of a vocabulary GEMM in tiles: waves of units times tiles per unit.
static int64_t split_cost(int m_tiles, int n_tiles, int sms, int s) {
  return cdiv(static_cast<int64_t>(m_tiles) * s, sms) * cdiv(n_tiles, s);
}

int dynamic_splits(int m_tiles, int n_tiles, int pairs) {
  // Pairs that draw their units from a counter balance the launch themselves, so the only
  // quantum left is one unit at the very end, and the pairs that share a W tile read it
  // within about half a unit's duration of each other: the shortest units (the most splits
  // the partials hold) give the least idle time and the fewest W re-reads.  Measured on the
  // 32K forward (same-process A/Bs with units drawn): 32 splits (units of about 25 tiles) took
  // 3.3 % less time than 10 (units of 79 tiles, whose last unit left most pairs idle for about
  // 1 ms); 64 splits (12 tiles) another 1.8 % (DRAM reads 19-20 -> 10.5-11.2 GB per launch).
  // A unit's start (a binary search in the row's sorted teacher ids, the hand-off of its
  // index) and end (three stores) are not free, though: units stay at least kMinUnitTiles
  // long (on a 22528-word vocabulary, 64 splits of 1-2 tiles kept the tensor pipe 87 % busy
  // against 90 % for 32), unless that leaves fewer than two units per pair.
  constexpr int kMinUnitTiles = 4;
  int s = (n_tiles + kMinUnitTiles - 1) / kMinUnitTiles;
  const int fill = static_cast<int>((2LL * pairs + m_tiles - 1) / m_tiles);
  if (s < fill) s = fill;
  if (s > n_tiles) s = n_tiles;
  return s < kMaxSplit ? s : kMaxSplit;
}

int plan_splits(int m_tiles, int n_tiles, int sms, int group) {
  // For launches whose units are dealt round-robin (the dS recompute, the one-SM forward):
  // pick the number of vocabulary splits per row block that minimises the critical path
  // (waves of units x tiles per unit).  At least sms/32 splits keep the row blocks in
  // flight at once (each re-read from L2 for every tile of its unit) to a few dozen.  With
  // units in groups of `group` row blocks, a count within 1 % of the best that makes a
  // group a whole number of waves is preferred: no wave then straddles two groups, which
  // would double the row blocks of A held in L2 (measured on the 32K forward, 16 or 10
  // splits instead of 13: 1.2-1.3 % faster).
  int lo = (sms + 31) / 32;
  if (lo > n_tiles) lo = n_tiles;
  if (lo < 1) lo = 1;
  int hi = n_tiles < kMaxDealtSplit ? n_tiles : kMaxDealtSplit;
  auto cost = [&](int s) { return split_cost(m_tiles, n_tiles, sms, s); };
  int best = lo;
  for (int s = lo; s <= hi; ++s)
    if (cost(s) < cost(best)) best = s;
  const int64_t rows = group < m_tiles ? group : m_tiles;
  if (rows <= 1 || (rows * best) % sms == 0) return best;
  int aligned = 0;
  for (int s = lo; s <= hi; ++s)
    if ((rows * s) % sms == 0 && 100 * cost(s) <= 101 * cost(best) && (aligned == 0 || cost(s) < cost(aligned)))
      aligned = s;
  return aligned ? aligned : best;
}

GemmShape make_shape(int64_t M, int64_t N, int64_t Kd, int bn, int nsplit, uint32_t* status,
                     int rows_per_unit) {
  GemmShape g;
  g.M = static_cast<int>(M);
  g.N = static_cast<int>(N);
  g.Kd = static_cast<int>(Kd);
  g.m_tiles = static_cast<int>(cdiv(M, rows_per_unit));
  g.n_tiles = static_cast<int>(cdiv(N, bn));
  g.k_blocks = static_cast<int>(cdiv(Kd, 64));
  g.nsplit = nsplit;
  g.num_units = g.m_tiles * nsplit;
  g.group_m = 1;
  g.a_box3d = 0;
  g.b_box3d = 0;
  g.split_from = g.num_units;
  g.ksplit = 1;
  g.kpart = nullptr;
  g.sched = nullptr;
  g.sched_base = 0;
  g.status = status;
  g.limit_ns = kWaitLimitNs;
  return g;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map with 128-byte swizzle; out-of-range elements of a box read as zero.
bool encode_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_mn3d(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_extent,
                     uint64_t row_stride_bytes, uint32_t tile_mn) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || mn_extent % 64 != 0 || tile_mn % 64 != 0) return false;
  const cuuint64_t dims[3] = {64, k_extent, mn_extent / 64};
  const cuuint64_t strides[2] = {row_stride_bytes, 128};
  const cuuint32_t box[3] = {64, 64, tile_mn / 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_mn3d_sw64(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_extent,
                          uint64_t row_stride_bytes, uint32_t tile_mn) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || mn_extent % 32 != 0 || tile_mn % 32 != 0) return false;
  const cuuint64_t dims[3] = {32, k_extent, mn_extent / 32};
  const cuuint64_t strides[2] = {row_stride_bytes, 64};
  const cuuint32_t box[3] = {32, 64, tile_mn / 32};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_bf16_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {32, 64};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// MN-major B map of the two-SM kernel for tile width bn: the 3-D one-box-per-half view when
// the extent allows, else per-atom 2-D boxes; 64-byte swizzle when a half is 96 wide.
static bool encode_b_mn_pair(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_extent,
                             uint64_t row_stride_bytes, int bn, bool allow3d, bool* box3d) {
  const bool sw64 = (bn / 2) % 64 != 0;
  *box3d = allow3d && (sw64 ? encode_map_mn3d_sw64(map, base, mn_extent, k_extent, row_stride_bytes, bn / 2)
                            : encode_map_mn3d(map, base, mn_extent, k_extent, row_stride_bytes, bn / 2));
  if (*box3d) return true;
  return sw64 ? encode_map_bf16_sw64(map, base, mn_extent, k_extent, row_stride_bytes)
              : encode_map_bf16(map, base, mn_extent, k_extent, row_stride_bytes, 64, 64);
}

// ---------------------------------------------------------------- device info
struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
};

static fkl_status device_info(DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static std::mutex mu;
  static DevInfo cache[128];
  static bool have[128] = {};
  if (dev < 0 || dev >= 128) return fail(FKL_ERR_UNSUPPORTED, "device index %d out of range", dev);
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
      DevInfo di;
      if ((e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
          (e = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
      cache[dev] = di;
      have[dev] = true;
    }
    *out = cache[dev];
  }
  if (out->major != 10 || out->minor != 3)
    return fail(FKL_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                out->major, out->minor);
  return FKL_OK;
}

// Row blocks per group in the unit order of the dS recompute and the teacher cache's passes
// (the forward takes fwd_group_rows below): units run split-major within a group, so the 76
// pairs running together cover 38 row blocks of about 2 vocabulary splits and share each W
// tile in L2.  Against row-major order (about 6 row blocks per W tile) grouping cut the DRAM
// reads of the 32K products 2-4x.  In same-process A/Bs groups of 19 were 0.3 % slower than
// 38 for the dS recompute at 32K and about 1 % slower for the teacher's passes at the production
// shape, and 76 was 7-8 % slower than 38 (76 row blocks of H no longer stay in L2).  dW and
// dH keep row-major order, in which each A block is read once.
constexpr int kGroupRows = 38;

int group_rows(int m_tiles) { return kGroupRows < m_tiles ? kGroupRows : m_tiles; }

// Row blocks per group for the forward, whose units are drawn from a counter.  A buffer
// that SMs re-read stays resident in L2 up to about 64 MB on a GB300, not the 126 MB of L2
// in all, whichever SMs read it (half of L2 serves any set of SMs).  A group's H blocks and
// the W tiles in flight must fit in that half, so the forward takes a quarter of the pair
// count (19 row blocks; the pairs running together then cover four whole vocabulary
// splits).  In a same-process sweep of 12-38 row blocks this read the least DRAM on every
// workload (per launch: 9.2 against 13.8-15.4 GB for 38 at the 32K shapes, 73-74 against
// 132-141 GB at 256K, 27-28 against 107-118 GB on the packed 64K x 4096 workload; counts
// that do not divide the pair count read more), and the forward took 2.0 % less time at
// 256K and 6.5 % less on the packed workload, the same at 8K and 32K.
int fwd_group_rows(int m_tiles, int pairs) {
  const int g = pairs >= 4 ? pairs / 4 : 1;
  return g < m_tiles ? g : m_tiles;
}

// Tile width along d for the dW and dH products: the width with the least estimated time,
// counting padded columns and the measured relative cost per column of each width on GB300
// (narrower tiles need more operand bytes per FLOP).
static int choose_bn_d(int64_t d, bool pair) {
  const int cand[3] = {256, 192, 128};
  const double cost1[3] = {1.0, 1.11, 1.4};   // one-SM kernel
  // Two-SM kernel: 192-wide tiles (96-wide MN-major B halves, 64-byte swizzle) measured ~23 %
  // slower per FLOP than 256-wide ones on GB300, so they win only when 256 pads far more.
  const double cost2[3] = {1.0, 1.23, 1.3};
  const double* cost = pair ? cost2 : cost1;
  int best = 256;
  double best_t = 1e300;
  for (int i = 0; i < 3; ++i) {
    const double t = static_cast<double>(cdiv(d, cand[i]) * cand[i]) * cost[i];
    if (t < best_t) { best_t = t; best = cand[i]; }
  }
  return best;
}

// Vocabulary tiles per backward slab, at most the dS buffer's width and at least half of it.
// A slab's three GEMMs run in waves of CTA pairs: dW in (slab tiles x d tiles) units and dH in
// (Ct/256 x d tiles) units of one tile each, the dS recompute in units of plan_splits.  A slab
// width whose dW unit count falls just past a whole number of waves leaves most pairs idle in
// the last one (47 tiles x 12 d tiles = 564 units on 76 pairs: 7.4 waves, run as 8), so the
// width is the one with the shortest critical path over all slabs, counted in 64-deep k-steps
// of a 256 x 256 tile, plus a fixed cost per slab for the three launches' ramp and the dH
// read-modify-write (about 0.2 ms at 32K tokens; measured: 44-tile slabs beat 47 by 1 % per
// step at 32K, with dW 5 % faster).
void choose_slab_width(Plan* p, int pairs) {
  if (p->T == 0 || pairs < 1) return;
  constexpr double kSlabFixedSteps = 600.0;
  const int bnd = choose_bn_d(p->d, true);
  const int64_t nd = cdiv(p->d, bnd), mt = cdiv(p->Ct, 256), kd = cdiv(p->d, 64), kt = cdiv(p->Ct, 64);
  const double bs = bnd / 256.0;
  auto slab = [&](int64_t wt) {
    const int s = plan_splits(static_cast<int>(mt), static_cast<int>(wt), pairs, group_rows(static_cast<int>(mt)));
    return static_cast<double>(split_cost(static_cast<int>(mt), static_cast<int>(wt), pairs, s) * kd) +
           static_cast<double>(cdiv(wt * nd, pairs) * kt) * bs +
           static_cast<double>(cdiv(mt * nd, pairs) * 4 * wt) * bs + kSlabFixedSteps;
  };
  const int64_t vt = cdiv(p->V, kVocabTile), mmax = p->Vmax / kVocabTile;
  int64_t best_m = mmax;
  double best = 1e300;
  for (int64_t m = mmax; m >= 1 && 2 * m >= mmax; --m) {
    const int64_t ns = cdiv(vt, m);
    const double c = static_cast<double>(ns - 1) * slab(m) + slab(vt - (ns - 1) * m);
    if (c < best) { best = c; best_m = m; }
  }
  p->Vc = best_m * kVocabTile;
  p->nslabs = cdiv(p->V, p->Vc);
}

// The units of a product's last wave, r = units mod pairs of them, would keep r pairs busy
// for a whole unit while the others wait.  Split each into pairs / r pieces along K instead
// (at least kKsplitMinBlocks k-blocks each, at most `slots` pieces in all): every pair then
// runs at most one piece in that wave, and a fixup adds each unit's pieces in a fixed order.
// Only for products with one tile per unit (dW, dH).  dH at 32K tokens: 1536 units on 76
// pairs, 20.2 waves run as 21, become 20 waves and a quarter.
void plan_ksplit(GemmShape* g, int pairs, float* kpart, int slots) {
  if (kpart == nullptr || pairs < 2 || g->nsplit != g->n_tiles) return;
  const int r = g->num_units % pairs;
  if (r == 0) return;
  int s = pairs / r;
  if (s * r > slots) s = slots / r;
  if (s > g->k_blocks / kKsplitMinBlocks) s = g->k_blocks / kKsplitMinBlocks;
  if (s < 2) return;
  g->split_from = g->num_units - r;
  g->ksplit = s;
  g->kpart = kpart;
}

// CTA pairs of the current device, for planning only (76, a GB300's, when none is visible).
static int planning_pairs() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      sms >= 2)
    return sms / 2;
  return 76;
}

static fkl_status check_options(const fkl_options* o, int64_t T) {
  if (o == nullptr) return FKL_OK;
  if (o->reserved != 0) return fail(FKL_ERR_INVALID_ARG, "fkl_options.reserved must be 0");
  if (o->accumulate < 0 || o->accumulate > 3) return fail(FKL_ERR_INVALID_ARG, "bad fkl_options.accumulate");
  const float c = o->div_param;
  switch (o->divergence) {
    case FKL_DIV_KL: case FKL_DIV_TV: break;
    case FKL_DIV_JSD:
      if (!(c > 0.f && c < 1.f)) return fail(FKL_ERR_INVALID_ARG, "FKL_DIV_JSD needs 0 < div_param < 1");
      break;
    case FKL_DIV_SKEW_KL:
      if (!(c >= 0.f && c < 1.f)) return fail(FKL_ERR_INVALID_ARG, "FKL_DIV_SKEW_KL needs 0 <= div_param < 1");
      break;
    case FKL_DIV_SKEW_RKL:
      if (!(c > 0.f && c <= 1.f)) return fail(FKL_ERR_INVALID_ARG, "FKL_DIV_SKEW_RKL needs 0 < div_param <= 1");
      break;
    default: return fail(FKL_ERR_INVALID_ARG, "bad fkl_options.divergence");
  }
  if (!aligned(o->student_topk_logits, 4))
    return fail(FKL_ERR_ALIGNMENT, "fkl_options.student_topk_logits must be 4-byte aligned");
  if (!aligned(o->global_count, 8)) return fail(FKL_ERR_ALIGNMENT, "fkl_options.global_count must be 8-byte aligned");
  if (o->normalization == FKL_NORM_TOKENS) return FKL_OK;
  if (o->normalization != FKL_NORM_SEQUENCES) return fail(FKL_ERR_INVALID_ARG, "bad fkl_options.normalization");
  if (o->num_seqs < 1 || o->num_seqs > (T > 0 ? T : 1))
    return fail(FKL_ERR_INVALID_ARG, "fkl_options.num_seqs must be in [1, max(T, 1)]");
  if (T > 0 && o->seq_ids == nullptr) return fail(FKL_ERR_INVALID_ARG, "fkl_options.seq_ids is NULL");
  if (!aligned(o->seq_ids, 4)) return fail(FKL_ERR_ALIGNMENT, "fkl_options.seq_ids must be 4-byte aligned");
  return FKL_OK;
}

// Token weights of the loss (and N, S in the header) for the options' normaliser.
static cudaError_t run_weights(const fkl_options* o, const uint8_t* mask, int64_t T, uint8_t* ws, const Plan& pl,
                               WsHeader* hdr, cudaStream_t st) {
  const bool per_seq = o != nullptr && o->normalization == FKL_NORM_SEQUENCES;
  return launch_weights(mask, per_seq ? o->seq_ids : nullptr, per_seq ? o->num_seqs : 1, per_seq ? 1 : 0, T,
                        reinterpret_cast<int*>(ws + pl.off_scnt), hdr, reinterpret_cast<float*>(ws + pl.off_wrow),
                        o != nullptr ? o->global_count : nullptr, st);
}

static fkl_status check_common(const uint16_t* H, const uint16_t* W, const int32_t* idx, const float* z,
                               int64_t T, int64_t d, int64_t V, int64_t K, float tau, int64_t chunk,
                               void* ws, size_t ws_bytes, Plan* plan, bool bf16_grads = false) {
  if (!make_plan(T, d, V, K, chunk, plan, bf16_grads))
    return fail(FKL_ERR_INVALID_ARG,
                "unsupported shape T=%lld d=%lld V=%lld K=%lld chunk=%lld (need 0<=T<2^31, d%%8==0, "
                "8<=d<2^20, 1<=V<=2^30, 1<=K<=1024, chunk>=1)",
                (long long)T, (long long)d, (long long)V, (long long)K, (long long)chunk);
  if (!(tau > 0.f) || !std::isfinite(tau)) return fail(FKL_ERR_INVALID_ARG, "tau must be finite and > 0");
  if (W == nullptr) return fail(FKL_ERR_INVALID_ARG, "W is NULL");
  if (T > 0 && (H == nullptr || idx == nullptr || z == nullptr))
    return fail(FKL_ERR_INVALID_ARG, "H, topk_idx and topk_logits must not be NULL");
  if (ws == nullptr) return fail(FKL_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(FKL_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (ws_bytes < plan->total)
    return fail(FKL_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, plan->total);
  if (!aligned(W, 16) || (H && !aligned(H, 16))) return fail(FKL_ERR_ALIGNMENT, "H and W must be 16-byte aligned");
  if ((idx && !aligned(idx, 4)) || (z && !aligned(z, 4)))
    return fail(FKL_ERR_ALIGNMENT, "topk_idx and topk_logits must be 4-byte aligned");
  return FKL_OK;
}

}  // namespace fkl

using namespace fkl;

extern "C" {

size_t fkl_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk) {
  Plan p;
  return make_plan(T, d, V, K, chunk, &p) ? p.total : 0;
}

int64_t fkl_backward_slabs(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk) {
  Plan p;
  if (!make_plan(T, d, V, K, chunk, &p)) return 0;
  choose_slab_width(&p, planning_pairs());
  return p.nt * p.nslabs;
}

const char* fkl_last_error(void) { return g_last_error.c_str(); }

const char* fkl_status_string(int status) {
  switch (status) {
    case FKL_OK: return "ok";
    case FKL_ERR_INVALID_ARG: return "invalid argument";
    case FKL_ERR_ALIGNMENT: return "misaligned pointer or dimension";
    case FKL_ERR_UNSUPPORTED: return "unsupported device";
    case FKL_ERR_WORKSPACE: return "workspace missing or too small";
    case FKL_ERR_CUDA: return "CUDA error";
    case FKL_ERR_BAD_TOPK_ID: return "teacher id outside [0, V)";
    case FKL_ERR_BAD_TOPK_ROW: return "teacher row without a finite logit";
    case FKL_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FKL_ERR_BAD_SEQ_ID: return "sequence id outside [0, num_seqs)";
    case FKL_ERR_TOPK_OVERFLOW: return "too many tied top-K candidates in a row";
    case FKL_ERR_BAD_COUNT: return "global count below the call's own count";
    default: return "unknown status";
  }
}

fkl_status fkl_forward(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                       const float* topk_logits, const uint8_t* mask, int64_t T, int64_t d,
                       int64_t V, int64_t K, float tau, int64_t chunk, float* loss, float* lse,
                       void* workspace, size_t ws_bytes, void* stream) {
  return fkl_forward_ex(H, W, topk_idx, topk_logits, mask, T, d, V, K, tau, chunk, nullptr, loss, lse, workspace,
                        ws_bytes, stream);
}

fkl_status fkl_forward_ex(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                          const float* topk_logits, const uint8_t* mask, int64_t T, int64_t d,
                          int64_t V, int64_t K, float tau, int64_t chunk, const fkl_options* opts,
                          float* loss, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  Plan pl;
  fkl_status s = check_common(H, W, topk_idx, topk_logits, T, d, V, K, tau, chunk, workspace, ws_bytes, &pl);
  if (s != FKL_OK) return s;
  if ((s = check_options(opts, T)) != FKL_OK) return s;
  if (loss == nullptr || (T > 0 && lse == nullptr)) return fail(FKL_ERR_INVALID_ARG, "loss and lse must not be NULL");
  if (!aligned(loss, 4) || (lse && !aligned(lse, 4))) return fail(FKL_ERR_ALIGNMENT, "loss and lse must be 4-byte aligned");
  DevInfo di;
  if ((s = device_info(&di)) != FKL_OK) return s;
  {
    const NamedPtr ptrs[] = {{H, "H"}, {W, "W"}, {topk_idx, "topk_idx"}, {topk_logits, "topk_logits"},
                             {mask, "mask"}, {loss, "loss"}, {lse, "lse"}, {workspace, "workspace"},
                             {opts ? opts->seq_ids : nullptr, "fkl_options.seq_ids"},
                             {opts ? opts->student_topk_logits : nullptr, "fkl_options.student_topk_logits"},
                             {opts ? opts->global_count : nullptr, "fkl_options.global_count"}};
    if ((s = static_cast<fkl_status>(check_device_memory(ptrs))) != FKL_OK) return s;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  int2* pairs = reinterpret_cast<int2*>(ws + pl.off_pairs);
  float* crow = reinterpret_cast<float*>(ws + pl.off_crow);
  float* part = reinterpret_cast<float*>(ws + pl.off_part);
  double* bsum = reinterpret_cast<double*>(ws + pl.off_bsum);
  int* bcnt = reinterpret_cast<int*>(ws + pl.off_bcnt);
  const float* wrow = reinterpret_cast<const float*>(ws + pl.off_wrow);

  const DivSpec dv{opts ? opts->divergence : FKL_DIV_KL, opts ? opts->div_param : 0.f};
  float* user_s = opts ? opts->student_topk_logits : nullptr;
  const bool record_s = dv.kind != FKL_DIV_KL || user_s != nullptr;
  int* slot = reinterpret_cast<int*>(ws + pl.off_slot);
  float* sg = reinterpret_cast<float*>(ws + pl.off_sg);

  if (T > 0) {
    if ((e = launch_prep(topk_idx, topk_logits, T, (int)K, (int)V, tau, pairs, slot, crow, &hdr->status, st)) !=
        cudaSuccess)
      return cuda_fail(e, "prep kernel");
    if ((e = run_weights(opts, mask, T, ws, pl, hdr, st)) != cudaSuccess) return cuda_fail(e, "weights kernels");
    // Two-SM tiles: each CTA of a pair loads 128 rows of H and 128 rows of the W tile.
    CUtensorMap mH, mW;
    if (!encode_map_bf16(&mH, H, d, T, d * 2, 64, 128) || !encode_map_bf16(&mW, W, d, V, d * 2, 64, kVocabTile / 2))
      return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for H or W");
    // Units drawn from a counter (the header was zeroed above: this is the call's first
    // dynamically scheduled launch, sched_base 0), in groups of row blocks, split-major.
    const int m_tiles = (int)cdiv(T, 256), n_tiles = (int)cdiv(V, kVocabTile);
    GemmShape g = make_shape(T, V, d, kVocabTile, dynamic_splits(m_tiles, n_tiles, di.sms / 2), &hdr->status, 256);
    g.group_m = fwd_group_rows(g.m_tiles, di.sms / 2);
    g.sched = &hdr->items_taken;
    const int nsplit = g.nsplit;
    FwdParams fp;
    fp.pairs = pairs;
    fp.part = part;
    fp.sg = record_s ? sg : nullptr;
    fp.T = (int)T; fp.K = (int)K; fp.V = (int)V; fp.nsplit = nsplit;
    fp.scale2 = kLog2e / tau;
    trace_launch_begin(st);
    if ((e = launch_gemm2_fwd(mH, mW, g, fp, di.sms, st)) != cudaSuccess) return cuda_fail(e, "forward GEMM");
    trace_launch_end(st, 0, 2.0 * T * V * d);
    if ((e = launch_combine_rows(part, nsplit, crow, wrow, T, tau, lse, bsum, bcnt, pl.nb, st)) != cudaSuccess)
      return cuda_fail(e, "combine kernel");
    if (record_s &&
        (e = launch_div_rows(dv, pairs, slot, sg, lse, wrow, T, (int)K, tau, user_s, bsum, bcnt, pl.nb, st)) !=
            cudaSuccess)
      return cuda_fail(e, "divergence kernel");
    if ((e = launch_combine_final(bsum, bcnt, T, pl.nb, tau, hdr, loss, st)) != cudaSuccess)
      return cuda_fail(e, "combine kernel");
  } else {
    if ((e = launch_combine(part, 1, crow, wrow, 0, tau, lse, bsum, bcnt, 0, hdr, loss, st)) != cudaSuccess)
      return cuda_fail(e, "combine kernels");
  }
  return FKL_OK;
}

// The fixup of a K-split product, traced (kind 4) right after the product it completes.
static cudaError_t run_fixup(int bn, const GemmShape& g, const F32Params& p, cudaStream_t st) {
  if (g.ksplit < 2) return cudaSuccess;
  trace_launch_begin(st);
  const cudaError_t e = launch_ksplit_fixup(bn, g, p, st);
  if (e == cudaSuccess) trace_launch_end(st, 4, 0.0);
  return e;
}

// Gradient outputs of one backward call: fp32 (dH, dW) or bf16 (dH16, dW16).
struct GradOut {
  bool bf16;
  float* dH;
  float* dW;
  uint16_t* dH16;
  uint16_t* dW16;
};

// Where the dW product of token block b writes slab rows [v0, v0 + w): the caller's fp32 dW
// (summed over token blocks in order), or, for bf16 gradients, fp32 sums in the workspace
// (several token blocks; all of dW, or the current slab's rows when slabs are the outer
// loop) that the last block adds to its tile and rounds to bf16.
static F32Params dw_output(const Plan& pl, const GradOut& out, int accum, float* wsum, int64_t b, int64_t v0,
                           int64_t w, int64_t d) {
  F32Params p;
  p.ldo = d; p.M = (int)w; p.N = (int)d;
  if (!out.bf16) {
    p.out = out.dW + v0 * d;
    p.accumulate = (b > 0 || (accum & FKL_ACCUMULATE_DW)) ? 1 : 0;
    p.vec_ok = aligned(out.dW, 32) ? 1 : 0;
    return p;
  }
  p.out = pl.nt == 1 ? nullptr : pl.slab_outer ? wsum : wsum + v0 * d;
  p.accumulate = b > 0 ? 1 : 0;
  p.vec_ok = 1;
  if (b == pl.nt - 1) {
    p.out16 = out.dW16 + v0 * d; p.ldo16 = d; p.vec16_ok = aligned(out.dW16, 16) ? 1 : 0;
  }
  return p;
}

// Where the dH product of slab j writes the rows [r0, r0 + rows) of its token block: the
// caller's fp32 dH (summed over slabs in order), or, for bf16 gradients, an fp32 sum in the
// workspace (the current block's rows, or all of dH when slabs are the outer loop) that the
// last slab adds to its tile and rounds to bf16.
static F32Params dh_output(const Plan& pl, const GradOut& out, int accum, float* hsum, int64_t j, int64_t r0,
                           int64_t rows, int64_t d) {
  F32Params p;
  p.ldo = d; p.M = (int)rows; p.N = (int)d;
  if (!out.bf16) {
    p.out = out.dH + r0 * d;
    p.accumulate = (j > 0 || (accum & FKL_ACCUMULATE_DH)) ? 1 : 0;
    p.vec_ok = aligned(out.dH, 32) ? 1 : 0;
    return p;
  }
  p.out = pl.slab_outer ? hsum + r0 * d : hsum;
  p.accumulate = j > 0 ? 1 : 0;
  p.vec_ok = 1;
  if (j == pl.nslabs - 1) {
    p.out16 = out.dH16 + r0 * d; p.ldo16 = d; p.vec16_ok = aligned(out.dH16, 16) ? 1 : 0;
  }
  return p;
}

// One block of the backward: token block b x vocabulary slab j (the dS recompute, its dW
// product and its dH product, each K-split fixup after its product).  All three products use
// two-SM tiles (256 rows per CTA pair, B split between the CTAs).
static fkl_status run_block(const Plan& pl, const DevInfo& di, const uint16_t* H, const uint16_t* W,
                           const float* lse, int64_t T, int64_t d, int64_t V, int64_t K, float tau,
                           const DivSpec& dv, int accum, uint8_t* ws, const GradOut& out, int64_t b, int64_t j,
                           cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  const int2* pairs = reinterpret_cast<const int2*>(ws + pl.off_pairs);
  const float* arow = reinterpret_cast<const float*>(ws + pl.off_arow);
  uint16_t* ds = reinterpret_cast<uint16_t*>(ws + pl.off_ds);
  float* kpart = reinterpret_cast<float*>(ws + pl.off_kpart);
  float* hsum = reinterpret_cast<float*>(ws + pl.off_hsum);  // bf16 gradients: dH sums over slabs
  float* wsum = reinterpret_cast<float*>(ws + pl.off_wsum);  // bf16 gradients: dW sums over token blocks
  cudaError_t e;
  const int bnd = choose_bn_d(d, true);
  const int64_t Vc = pl.Vc;
  const float* wrow = reinterpret_cast<const float*>(ws + pl.off_wrow);
  const int64_t r0 = b * pl.Ct;
  const int64_t rows = (T - r0) < pl.Ct ? (T - r0) : pl.Ct;
  const uint16_t* Hb = H + r0 * d;
  CUtensorMap mH_k, mH_mn;
  bool h3d = false;
  if (!encode_map_bf16(&mH_k, Hb, d, rows, d * 2, 64, 128) || !encode_b_mn_pair(&mH_mn, Hb, d, rows, d * 2, bnd, true, &h3d))
    return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for H block %lld", (long long)b);
  const int64_t v0 = j * Vc;
  const int64_t w = (V - v0) < Vc ? (V - v0) : Vc;
  const uint16_t* Wj = W + v0 * d;
  CUtensorMap mW_k, mW_mn, mD_mn, mD_k;
  // The dS buffer holds zeros in the columns [w, round_up(w, 256)) of every row, so its
  // 3-D view may span round_up(w, 64) columns.
  bool w3d = false;
  const bool wmap = encode_b_mn_pair(&mW_mn, Wj, d, w, d * 2, bnd, true, &w3d);
  const bool d3d = encode_map_mn3d(&mD_mn, ds, cdiv(w, 64) * 64, rows, Vc * 2, 128);
  if (!encode_map_bf16(&mW_k, Wj, d, w, d * 2, 64, kVocabTile / 2) || !wmap ||
      (!d3d && !encode_map_bf16(&mD_mn, ds, w, rows, Vc * 2, 64, 64)) ||
      !encode_map_bf16(&mD_k, ds, w, rows, Vc * 2, 64, 128))
    return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for block (%lld, %lld)", (long long)b, (long long)j);

  // dS[block] = g tau w_t (q - ptilde), recomputing S = H_block W_slab^T.
  const int m_tiles = (int)cdiv(rows, 256), n_tiles = (int)cdiv(w, kVocabTile);
  GemmShape g3 = make_shape(rows, w, d, kVocabTile, plan_splits(m_tiles, n_tiles, di.sms / 2, group_rows(m_tiles)),
                            &hdr->status, 256);
  g3.group_m = group_rows(g3.m_tiles);
  DsParams dp;
  dp.pairs = pairs + r0 * K; dp.lse = lse + r0; dp.wrow = wrow + r0;
  dp.arow = dv.kind != FKL_DIV_KL ? arow + r0 : nullptr;
  dp.hdr = hdr; dp.ds = ds; dp.ld_ds = Vc;
  dp.T = (int)rows; dp.K = (int)K; dp.V = (int)V; dp.v0 = (int)v0; dp.slab_w = (int)w;
  dp.scale2 = kLog2e / tau;
  const double block_flops = 2.0 * rows * w * d;
  trace_launch_begin(st);
  if ((e = launch_gemm2_ds(mH_k, mW_k, g3, dp, di.sms, st)) != cudaSuccess) return cuda_fail(e, "dS GEMM");
  trace_launch_end(st, 1, block_flops);

  // dW[slab] (+)= dS[block]^T H_block  (token blocks in order).
  GemmShape g4 = make_shape(w, d, rows, bnd, (int)cdiv(d, bnd), &hdr->status, 256);
  g4.a_box3d = d3d ? 1 : 0;
  g4.b_box3d = h3d ? 1 : 0;
  const F32Params p4 = dw_output(pl, out, accum, wsum, b, v0, w, d);
  plan_ksplit(&g4, di.sms / 2, kpart, kKsplitSlots);
  trace_launch_begin(st);
  if ((e = launch_gemm2_f32(bnd, true, true, mD_mn, mH_mn, g4, p4, di.sms, st)) != cudaSuccess)
    return cuda_fail(e, "dW GEMM");
  trace_launch_end(st, 2, block_flops);
  if ((e = run_fixup(bnd, g4, p4, st)) != cudaSuccess) return cuda_fail(e, "dW K-split fixup");

  // dH[block] (+)= dS[block] W[slab]  (slabs in order).
  GemmShape g5 = make_shape(rows, d, w, bnd, (int)cdiv(d, bnd), &hdr->status, 256);
  g5.b_box3d = w3d ? 1 : 0;
  const F32Params p5 = dh_output(pl, out, accum, hsum, j, r0, rows, d);
  plan_ksplit(&g5, di.sms / 2, kpart, kKsplitSlots);
  trace_launch_begin(st);
  if ((e = launch_gemm2_f32(bnd, false, true, mD_k, mW_mn, g5, p5, di.sms, st)) != cudaSuccess)
    return cuda_fail(e, "dH GEMM");
  trace_launch_end(st, 3, block_flops);
  if ((e = run_fixup(bnd, g5, p5, st)) != cudaSuccess) return cuda_fail(e, "dH K-split fixup");
  return FKL_OK;
}

// The backward's GEMMs, after the light kernels have prepared the pairs, the token weights
// and the scales in the workspace: blocks of Ct tokens x Vc vocabulary columns, token blocks
// outer (slabs outer for bf16 gradients when the plan says so; the same summation orders).
// dW of a slab accumulates over the token blocks and dH of a token block over the slabs, both
// in a fixed order (deterministic).
static fkl_status run_backward_blocks(const Plan& pl, const DevInfo& di, const uint16_t* H, const uint16_t* W,
                                      const float* lse, int64_t T, int64_t d, int64_t V, int64_t K, float tau,
                                      const DivSpec& dv, int accum, uint8_t* ws, const GradOut& out,
                                      cudaStream_t st) {
  const int64_t outer = pl.slab_outer ? pl.nslabs : pl.nt, inner = pl.slab_outer ? pl.nt : pl.nslabs;
  for (int64_t o = 0; o < outer; ++o)
    for (int64_t n = 0; n < inner; ++n) {
      const int64_t b = pl.slab_outer ? n : o, j = pl.slab_outer ? o : n;
      const fkl_status s = run_block(pl, di, H, W, lse, T, d, V, K, tau, dv, accum, ws, out, b, j, st);
      if (s != FKL_OK) return s;
    }
  return FKL_OK;
}

fkl_status fkl_backward(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                        const float* topk_logits, const uint8_t* mask, const float* lse,
                        const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K,
                        float tau, int64_t chunk, float* dH, float* dW, void* workspace,
                        size_t ws_bytes, void* stream) {
  return fkl_backward_ex(H, W, topk_idx, topk_logits, mask, lse, grad_loss, T, d, V, K, tau, chunk, nullptr, dH, dW,
                         workspace, ws_bytes, stream);
}

// The backward of both entry points: fp32 gradients (fkl_backward_ex) or bf16 ones
// (fkl_backward_bf16), which need the fp32 sums laid out by make_plan(bf16_grads).
static fkl_status backward_impl(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                                const float* topk_logits, const uint8_t* mask, const float* lse,
                                const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K, float tau,
                                int64_t chunk, const fkl_options* opts, const GradOut& out, void* workspace,
                                size_t ws_bytes, void* stream) {
  g_last_error.clear();
  Plan pl;
  fkl_status s = check_common(H, W, topk_idx, topk_logits, T, d, V, K, tau, chunk, workspace, ws_bytes, &pl,
                              out.bf16);
  if (s != FKL_OK) return s;
  if ((s = check_options(opts, T)) != FKL_OK) return s;
  const int accum = opts ? opts->accumulate : 0;
  if (out.bf16 && accum != 0)
    return fail(FKL_ERR_INVALID_ARG, "bf16 gradients do not accumulate (fkl_options.accumulate must be 0)");
  const void* gH = out.bf16 ? static_cast<const void*>(out.dH16) : static_cast<const void*>(out.dH);
  const void* gW = out.bf16 ? static_cast<const void*>(out.dW16) : static_cast<const void*>(out.dW);
  if (gW == nullptr || (T > 0 && (gH == nullptr || lse == nullptr)))
    return fail(FKL_ERR_INVALID_ARG, "dH, dW and lse must not be NULL");
  const DivSpec dv{opts ? opts->divergence : FKL_DIV_KL, opts ? opts->div_param : 0.f};
  if (dv.kind != FKL_DIV_KL && T > 0 && opts->student_topk_logits == nullptr)
    return fail(FKL_ERR_INVALID_ARG, "this divergence's backward needs fkl_options.student_topk_logits");
  if (!aligned(gW, 16) || (gH && !aligned(gH, 16))) return fail(FKL_ERR_ALIGNMENT, "dH and dW must be 16-byte aligned");
  if ((lse && !aligned(lse, 4)) || (grad_loss && !aligned(grad_loss, 4)))
    return fail(FKL_ERR_ALIGNMENT, "lse and grad_loss must be 4-byte aligned");
  DevInfo di;
  if ((s = device_info(&di)) != FKL_OK) return s;
  {
    const NamedPtr ptrs[] = {{H, "H"}, {W, "W"}, {topk_idx, "topk_idx"}, {topk_logits, "topk_logits"},
                             {mask, "mask"}, {lse, "lse"}, {grad_loss, "grad_loss"}, {gH, "dH"}, {gW, "dW"},
                             {workspace, "workspace"}, {opts ? opts->seq_ids : nullptr, "fkl_options.seq_ids"},
                             {opts ? opts->student_topk_logits : nullptr, "fkl_options.student_topk_logits"},
                             {opts ? opts->global_count : nullptr, "fkl_options.global_count"}};
    if ((s = static_cast<fkl_status>(check_device_memory(ptrs))) != FKL_OK) return s;
  }
  choose_slab_width(&pl, di.sms / 2);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  if (T == 0) {
    const size_t bytes = static_cast<size_t>(V) * d * (out.bf16 ? 2 : 4);
    if (!(accum & FKL_ACCUMULATE_DW) && (e = cudaMemsetAsync(const_cast<void*>(gW), 0, bytes, st)) != cudaSuccess)
      return cuda_fail(e, "cudaMemsetAsync(dW)");
    return FKL_OK;
  }
  int2* pairs = reinterpret_cast<int2*>(ws + pl.off_pairs);
  float* crow = reinterpret_cast<float*>(ws + pl.off_crow);
  int* slot = reinterpret_cast<int*>(ws + pl.off_slot);
  float* arow = reinterpret_cast<float*>(ws + pl.off_arow);
  if ((e = launch_prep(topk_idx, topk_logits, T, (int)K, (int)V, tau, pairs, slot, crow, &hdr->status, st)) !=
      cudaSuccess)
    return cuda_fail(e, "prep kernel");
  if ((e = run_weights(opts, mask, T, ws, pl, hdr, st)) != cudaSuccess) return cuda_fail(e, "weights kernels");
  if ((e = launch_grad_scale(grad_loss, tau, hdr, st)) != cudaSuccess) return cuda_fail(e, "scale kernel");
  if (dv.kind != FKL_DIV_KL &&
      (e = launch_div_coef(dv, pairs, slot, opts->student_topk_logits, lse, T, (int)K, tau, arow, st)) != cudaSuccess)
    return cuda_fail(e, "divergence kernel");

  if ((s = run_backward_blocks(pl, di, H, W, lse, T, d, V, K, tau, dv, accum, ws, out, st)) != FKL_OK) return s;
  e = out.bf16 ? launch_poison16(out.dH16, T * d, out.dW16, V * d, &hdr->status, di.sms, st)
               : launch_poison(out.dH, T * d, out.dW, V * d, &hdr->status, di.sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "poison kernel");
  return FKL_OK;
}

fkl_status fkl_backward_ex(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                           const float* topk_logits, const uint8_t* mask, const float* lse,
                           const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K,
                           float tau, int64_t chunk, const fkl_options* opts, float* dH, float* dW,
                           void* workspace, size_t ws_bytes, void* stream) {
  return backward_impl(H, W, topk_idx, topk_logits, mask, lse, grad_loss, T, d, V, K, tau, chunk, opts,
                       GradOut{false, dH, dW, nullptr, nullptr}, workspace, ws_bytes, stream);
}

fkl_status fkl_backward_bf16(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                             const float* topk_logits, const uint8_t* mask, const float* lse,
                             const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K, float tau,
                             int64_t chunk, const fkl_options* opts, uint16_t* dH, uint16_t* dW,
                             void* workspace, size_t ws_bytes, void* stream) {
  return backward_impl(H, W, topk_idx, topk_logits, mask, lse, grad_loss, T, d, V, K, tau, chunk, opts,
                       GradOut{true, nullptr, nullptr, dH, dW}, workspace, ws_bytes, stream);
}

size_t fkl_backward_bf16_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk) {
  Plan p;
  return make_plan(T, d, V, K, chunk, &p, true) ? p.total : 0;
}

fkl_status fkl_read_status(const void* workspace, void* stream) {
  g_last_error.clear();
  if (workspace == nullptr) return fail(FKL_ERR_WORKSPACE, "workspace is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  if (h & kStatusBadIdBit) return FKL_ERR_BAD_TOPK_ID;
  if (h & kStatusBadRowBit) return FKL_ERR_BAD_TOPK_ROW;
  if (h & kStatusBadSeqBit) return FKL_ERR_BAD_SEQ_ID;
  if (h & kStatusTopkOverflowBit) return FKL_ERR_TOPK_OVERFLOW;
  if (h & kStatusBadCountBit) return FKL_ERR_BAD_COUNT;
  if (h & kStatusTimeoutBit) return FKL_ERR_TIMEOUT;
  return FKL_OK;
}

fkl_status fkl_local_count(const uint8_t* mask, int64_t T, const fkl_options* opts, int64_t* count,
                           void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (T < 0 || T >= (int64_t{1} << 31)) return fail(FKL_ERR_INVALID_ARG, "T must be in [0, 2^31)");
  fkl_status s = check_options(opts, T);
  if (s != FKL_OK) return s;
  if (count == nullptr) return fail(FKL_ERR_INVALID_ARG, "count must not be NULL");
  if (!aligned(count, 8)) return fail(FKL_ERR_ALIGNMENT, "count must be 8-byte aligned");
  if (workspace == nullptr) return fail(FKL_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(workspace, 256)) return fail(FKL_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  const size_t need = 256 + 4 * static_cast<size_t>(T > 0 ? T : 1);
  if (ws_bytes < need) return fail(FKL_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", ws_bytes, need);
  DevInfo di;
  if ((s = device_info(&di)) != FKL_OK) return s;
  {
    const NamedPtr ptrs[] = {{mask, "mask"}, {count, "count"}, {workspace, "workspace"},
                             {opts ? opts->seq_ids : nullptr, "fkl_options.seq_ids"}};
    if ((s = static_cast<fkl_status>(check_device_memory(ptrs))) != FKL_OK) return s;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  const bool per_seq = opts != nullptr && opts->normalization == FKL_NORM_SEQUENCES;
  if ((e = launch_local_count(mask, per_seq ? opts->seq_ids : nullptr, per_seq ? opts->num_seqs : 1, per_seq ? 1 : 0,
                              T, reinterpret_cast<int*>(ws + 256), reinterpret_cast<WsHeader*>(ws), count, st)) !=
      cudaSuccess)
    return cuda_fail(e, "count kernels");
  return FKL_OK;
}

fkl_status fkl_test_gemm(const uint16_t* A, const uint16_t* B, float* D, int64_t M, int64_t N,
                         int64_t Kd, int a_mn_major, int b_mn_major, int bn, int accumulate,
                         void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!A || !B || !D) return fail(FKL_ERR_INVALID_ARG, "A, B and D must not be NULL");
  if (M < 1 || N < 1 || Kd < 1 || M >= (1 << 30) || N >= (1 << 30) || Kd >= (1 << 30))
    return fail(FKL_ERR_INVALID_ARG, "M, N, Kd must be in [1, 2^30)");
  if (bn != 256 && bn != 192 && bn != 128) return fail(FKL_ERR_INVALID_ARG, "bn must be 256, 192 or 128");
  const bool pair = (accumulate & 4) != 0;

  const int64_t a_inner = a_mn_major ? M : Kd, b_inner = b_mn_major ? N : Kd;
  if (a_inner % 8 != 0 || b_inner % 8 != 0)
    return fail(FKL_ERR_ALIGNMENT, "the contiguous extent of A and B must be a multiple of 8");
  if (!aligned(A, 16) || !aligned(B, 16) || !aligned(D, 4)) return fail(FKL_ERR_ALIGNMENT, "misaligned A, B or D");
  if (!workspace || ws_bytes < 256) return fail(FKL_ERR_WORKSPACE, "workspace needs 256 bytes");
  if (!aligned(workspace, 256)) return fail(FKL_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  DevInfo di;
  fkl_status s = device_info(&di);
  if (s != FKL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace header)");
  // MN-major operands use one 3-D box per tile when their extent is a multiple of 64, unless
  // bit 1 of `accumulate` asks for the 64-wide 2-D boxes.
  const bool allow3d = (accumulate & 2) == 0;
  CUtensorMap mA, mB;
  const uint32_t b_tile = pair ? (uint32_t)bn / 2 : (uint32_t)bn;  // B rows / columns per CTA
  const bool a3d = a_mn_major && allow3d && encode_map_mn3d(&mA, A, M, Kd, M * 2, 128);
  bool b3d = false;
  bool ok = a3d || (a_mn_major ? encode_map_bf16(&mA, A, M, Kd, M * 2, 64, 64) : encode_map_bf16(&mA, A, Kd, M, Kd * 2, 64, 128));
  if (b_mn_major && pair) {
    ok = ok && encode_b_mn_pair(&mB, B, N, Kd, N * 2, bn, allow3d, &b3d);
  } else {
    b3d = b_mn_major && allow3d && encode_map_mn3d(&mB, B, N, Kd, N * 2, b_tile);
    ok = ok && (b3d || (b_mn_major ? encode_map_bf16(&mB, B, N, Kd, N * 2, 64, 64)
                                   : encode_map_bf16(&mB, B, Kd, N, Kd * 2, 64, b_tile)));
  }
  if (!ok) return fail(FKL_ERR_CUDA, "cuTensorMapEncodeTiled failed for A or B");
  GemmShape g = make_shape(M, N, Kd, bn, (int)cdiv(N, bn), &hdr->status, pair ? 256 : 128);
  g.a_box3d = a3d ? 1 : 0;
  g.b_box3d = b3d ? 1 : 0;
  F32Params p;
  p.out = D; p.ldo = N; p.M = (int)M; p.N = (int)N; p.accumulate = (accumulate & 1) ? 1 : 0;
  p.vec_ok = (N % 8 == 0 && aligned(D, 32)) ? 1 : 0;
  if (pair && (accumulate & 8)) {
    const int slots = static_cast<int>((ws_bytes - 256) / (static_cast<size_t>(256) * bn * 4));
    plan_ksplit(&g, di.sms / 2, reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256),
                slots < kKsplitSlots ? slots : kKsplitSlots);
  }
  e = pair ? launch_gemm2_f32(bn, a_mn_major != 0, b_mn_major != 0, mA, mB, g, p, di.sms, st)
           : launch_gemm_f32(bn, a_mn_major != 0, b_mn_major != 0, mA, mB, g, p,
                             g.num_units < di.sms ? g.num_units : di.sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "test GEMM");
  if ((e = launch_ksplit_fixup(bn, g, p, st)) != cudaSuccess) return cuda_fail(e, "test GEMM K-split fixup");
  return FKL_OK;
}

fkl_status fkl_test_backward_plan(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk, int32_t sms,
                                  int64_t* out) {
  g_last_error.clear();
  if (out == nullptr) return fail(FKL_ERR_INVALID_ARG, "out is NULL");
  if (sms < 2) return fail(FKL_ERR_INVALID_ARG, "sms must be at least 2");
  Plan pl;
  if (!make_plan(T, d, V, K, chunk, &pl)) return fail(FKL_ERR_INVALID_ARG, "unsupported shape");
  choose_slab_width(&pl, sms / 2);
  out[0] = pl.Ct;
  out[1] = pl.nt;
  out[2] = pl.Vc;
  out[3] = pl.nslabs;
  out[4] = pl.Vmax;
  return FKL_OK;
}

fkl_status fkl_test_wait_timeout(uint64_t limit_ns, void* workspace, size_t ws_bytes, void* stream) {
  g_last_error.clear();
  if (!workspace || ws_bytes < 256) return fail(FKL_ERR_WORKSPACE, "workspace needs 256 bytes");
  if (!aligned(workspace, 256)) return fail(FKL_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  if (limit_ns == 0 || limit_ns > 1000000000ull) return fail(FKL_ERR_INVALID_ARG, "limit_ns must be in (0, 1e9]");
  DevInfo di;
  fkl_status s = device_info(&di);
  if (s != FKL_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(workspace, 0, 256, st);
  if (e == cudaSuccess) e = launch_wait_timeout_test(static_cast<uint32_t*>(workspace), limit_ns, st);
  if (e != cudaSuccess) return cuda_fail(e, "timeout probe");
  return FKL_OK;
}

}  // extern "C"
