// Declarations shared by the translation units of the fused chunked KL library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace fkl {

// Bits of the device status word (first 4 bytes of the workspace).
constexpr uint32_t kStatusBadIdBit = 1u;
constexpr uint32_t kStatusBadRowBit = 2u;
constexpr uint32_t kStatusTimeoutBit = 4u;
constexpr uint32_t kStatusBadSeqBit = 8u;
constexpr uint32_t kStatusTopkOverflowBit = 16u;
constexpr uint32_t kStatusBadCountBit = 32u;

// Workspace header (first 256 bytes): status word, valid tokens, sequences with a valid
// token, g * tau (the backward's dS scale is g * tau * w_t), and the counter from which the
// dynamically scheduled GEMM launches of one call draw their work items.
struct WsHeader {
  uint32_t status;
  int32_t n_valid;
  int32_t n_seqs;
  float gtau;
  int32_t items_taken;  // work-item counter of the dynamically scheduled GEMM launches
};

constexpr int kVocabTile = 256;                   // tile width of the vocabulary axis
constexpr int kMaxSplit = 64;                     // most vocabulary splits per row block (partials)
constexpr int kMaxDealtSplit = 32;                // most splits of a launch whose units are dealt round-robin
constexpr int64_t kMaxTokenBlocks = 64;           // most token blocks of the backward
constexpr uint64_t kWaitLimitNs = 5000000000ull;  // per pipeline wait
constexpr float kLog2e = 1.4426950408889634f;      // log2(e): natural-log scale to base 2
constexpr float kLn2 = 0.69314718055994531f;       // ln(2): base-2 log back to natural

// Where each buffer lives inside the caller's workspace, and the backward's blocks.
struct Plan {
  int64_t T, d, V, K, chunk;
  int64_t Ct;      // tokens per backward block (T, or a multiple of 256 below it)
  int64_t nt;      // token blocks of the backward
  int64_t Vc;      // vocabulary columns per backward slab (multiple of kVocabTile)
  int64_t Vmax;    // widest slab the dS buffer holds (Vc <= Vmax)
  int64_t nslabs;  // vocabulary slabs of the backward
  bool slab_outer; // bf16 gradients with several token blocks: slabs in the outer loop
  int64_t nb;      // row blocks of the combine step (256 rows each)
  size_t off_pairs, off_crow, off_wrow, off_scnt, off_part, off_bsum, off_bcnt, off_ds;
  size_t off_slot;  // int32 [T][K]: original slot of each sorted pair
  size_t off_sg;    // fp32 [T][K]: student logit at each sorted pair (other divergences)
  size_t off_arow;  // fp32 [T]: per-row factor a_t of dS (other divergences)
  size_t off_kpart; // fp32 partial tiles of K-split dW / dH units
  // bf16 gradients only: fp32 sums of dH over slabs and of dW over token blocks.  Token
  // blocks outer: dH of the current block [Ct][d] and all of dW [V][d]; slabs outer (when
  // that needs less): all of dH [T][d] and dW of the current slab [Vmax][d].
  size_t off_hsum;
  size_t off_wsum;
  size_t total;
};

// Divergence of the loss (the FKL_DIV_* values of fkl.h) and its parameter.
struct DivSpec {
  int kind;
  float param;
};

// Sets the message that fkl_last_error() returns on the calling thread.
void set_last_error_message(const char* msg);

// A pointer argument and its name, for check_device_memory.
struct NamedPtr {
  const void* p;
  const char* name;
};
// Every pointer that the kernels or the tensor maps will dereference must be device (or
// managed) memory of the current device.  A host pointer given by mistake is refused here,
// before anything is enqueued, instead of faulting in a kernel.  NULL entries pass (whether
// an argument may be NULL is checked by each entry point).  FKL_OK or FKL_ERR_INVALID_ARG
// (with the argument's name in fkl_last_error()); int for the fkl_status values of fkl.h.
int check_device_memory(const NamedPtr* ptrs, int n);
template <int N>
int check_device_memory(const NamedPtr (&ptrs)[N]) {
  return check_device_memory(ptrs, N);
}

// Event pair around one GEMM launch when a trace is active on this thread (fkl_trace.cu).
// kind: 0 forward, 1 dS recompute, 2 dW, 3 dH.
void trace_launch_begin(cudaStream_t st);
void trace_launch_end(cudaStream_t st, int kind, double flops);

// bf16_grads: also lay out the fp32 sums that bf16 gradient outputs need (fkl_backward_bf16).
// max_splits: vocabulary splits the forward's partials hold per row.
bool make_plan(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk, Plan* p, bool bf16_grads = false,
               int max_splits = kMaxSplit);

// Vocabulary splits per 128-row block for a persistent launch over m_tiles x n_tiles.
// group: row blocks per group of the unit order (1 = row-major).
int plan_splits(int m_tiles, int n_tiles, int sms, int group = 1);
// Vocabulary splits per row block for a dynamically scheduled launch (GemmShape::sched) over
// m_tiles x n_tiles on `pairs` CTA pairs.
int dynamic_splits(int m_tiles, int n_tiles, int pairs);
// Sets p->Vc and p->nslabs for a device with `pairs` CTA pairs (see fkl_api.cu).
void choose_slab_width(Plan* p, int pairs);

// ---------------------------------------------------------------- small kernels
cudaError_t launch_prep(const int32_t* idx, const float* logits, int64_t T, int K, int V, float tau,
                        int2* pairs, int* slot, float* crow, uint32_t* status, cudaStream_t st);
// Forward, after the combine has written lse: for a divergence other than KL, D_t of every
// row from the sorted pairs and the student logits sg at them, and the per-block sums of
// w_t D_t (overwriting the combine's KL sums); then, if user_s is not NULL, the student
// logits scattered to the caller's slot order.  Call launch_combine_final afterwards.
cudaError_t launch_div_rows(DivSpec dv, const int2* pairs, const int* slot, const float* sg,
                            const float* lse, const float* wrow, int64_t T, int K, float tau,
                            float* user_s, double* bsum, int* bcnt, int64_t nb, cudaStream_t st);
// Backward, after prep: a_t into arow and, in place of p in the pairs, the per-id term r so
// that dS = g tau w_t (a_t q - r) reproduces the divergence's gradient.
cudaError_t launch_div_coef(DivSpec dv, int2* pairs, const int* slot, const float* user_s,
                            const float* lse, int64_t T, int K, float tau, float* arow, cudaStream_t st);
// Token weights w_t into wrow[T] (and N, S into the header); seq may be NULL (one sequence).
// global_count (device, may be NULL): the whole batch's count (N, or S per_sequence) in place
// of this call's own; a value below the call's own count sets kStatusBadCountBit.
cudaError_t launch_weights(const uint8_t* mask, const int32_t* seq, int num_seqs, int per_sequence,
                           int64_t T, int* cnt, WsHeader* hdr, float* wrow, const int64_t* global_count,
                           cudaStream_t st);
// This call's own count (N, or S per_sequence) into *count; cnt holds num_seqs ints of scratch.
cudaError_t launch_local_count(const uint8_t* mask, const int32_t* seq, int num_seqs, int per_sequence,
                               int64_t T, int* cnt, WsHeader* hdr, int64_t* count, cudaStream_t st);
// lse_t and the per-block sums of w_t KL_t (launch_combine_rows), then the loss from the
// block sums (launch_combine_final); launch_combine runs both.
cudaError_t launch_combine_rows(const float* part, int nsplit, const float* crow, const float* wrow,
                                int64_t T, float tau, float* lse, double* bsum, int* bcnt, int64_t nb,
                                cudaStream_t st);
cudaError_t launch_combine_final(const double* bsum, const int* bcnt, int64_t T, int64_t nb, float tau,
                                 WsHeader* hdr, float* loss, cudaStream_t st);
cudaError_t launch_combine(const float* part, int nsplit, const float* crow, const float* wrow,
                           int64_t T, float tau, float* lse, double* bsum, int* bcnt, int64_t nb,
                           WsHeader* hdr, float* loss, cudaStream_t st);
cudaError_t launch_grad_scale(const float* grad, float tau, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_poison(float* a, int64_t na, float* b, int64_t nb, const uint32_t* status,
                          int sms, cudaStream_t st);
// The same for bf16 gradients (NaN = 0x7FC0).
cudaError_t launch_poison16(uint16_t* a, int64_t na, uint16_t* b, int64_t nb, const uint32_t* status,
                            int sms, cudaStream_t st);
cudaError_t launch_wait_timeout_test(uint32_t* status, uint64_t limit_ns, cudaStream_t st);

// ---------------------------------------------------------------- GEMMs
// Problem of one persistent tcgen05 GEMM launch: D[M, N] = A[M, Kd] * B[N, Kd]^T in
// 128 x BN tiles.  A unit is one 128-row block and a contiguous range of n tiles.
struct GemmShape {
  int M, N, Kd;
  int m_tiles, n_tiles, k_blocks;
  int nsplit;     // units per row block
  int num_units;  // m_tiles * nsplit
  int group_m;    // row blocks per group: units run split-major within a group (1 = row-major)
  int a_box3d;    // MN-major A loaded by one 3-D box per tile (else 64-wide 2-D boxes)
  int b_box3d;    // same for B
  // Units from split_from on (those of the last, partial wave) are split along K into ksplit
  // pieces; each piece stores its fp32 partial tile in kpart, and a fixup kernel adds the
  // pieces in order (fp32 products, two-SM kernel only; split_from = num_units: none).
  int split_from;
  int ksplit;
  float* kpart;  // [(unit - split_from) * ksplit + piece][256][bn]
  // Dynamic scheduling (two-SM kernel; NULL: items dealt round-robin).  Each pair starts on
  // item `cluster`, then draws the next from *sched: item = pairs + (*sched)++ - sched_base.
  // A launch advances *sched by exactly its number of items, so consecutive launches of one
  // call give each the running total as sched_base (the counter is zeroed with the header).
  int* sched;
  int sched_base;
  uint32_t* status;
  uint64_t limit_ns;
};

// Partial tiles the workspace holds for K-split units (256 x 256 fp32 each).
constexpr int kKsplitSlots = 80;
// Fewest 64-deep k-blocks per K piece.
constexpr int kKsplitMinBlocks = 4;
// Splits the units of the last, partial wave of a one-tile-per-unit fp32 product along K
// (see fkl_api.cu); leaves the shape unsplit when that does not pay.
void plan_ksplit(GemmShape* g, int pairs, float* kpart, int slots);

// Row blocks per group of the unit order for products over the vocabulary (see fkl_api.cu).
int group_rows(int m_tiles);
// Row blocks per group of the forward's drawn units (see fkl_api.cu).
int fwd_group_rows(int m_tiles, int pairs);

// rows_per_unit: 128 for the one-SM kernel, 256 for the two-SM (CTA pair) kernel.
GemmShape make_shape(int64_t M, int64_t N, int64_t Kd, int bn, int nsplit, uint32_t* status,
                     int rows_per_unit = 128);

// Forward: online base-2 logsumexp and top-K gather per (row, vocabulary split).
struct FwdParams {
  const int2* pairs;  // [T][K] (id, p) sorted by id
  float* part;        // [3][nsplit][T]: running max (base 2), sum, gather
  float* sg;          // [T][K] student logit at each sorted pair, or NULL (not recorded)
  int T, K, V, nsplit;
  float scale2;       // log2(e) / tau
};

// Backward recompute: dS = g tau w_t (a_t q - r) for one block (a range of T tokens x a
// vocabulary slab of slab_w columns from v0), bf16, with r the pairs' second field added
// at their ids (KL: a_t = 1, r = p, i.e. q - ptilde).  The per-token pointers start at the
// block's first token.
struct DsParams {
  const int2* pairs;
  const float* lse;
  const float* wrow;  // w_t (0 for masked tokens)
  const float* arow;  // a_t, or NULL for a_t = 1
  const WsHeader* hdr;
  uint16_t* ds;       // [T][ld_ds]
  int64_t ld_ds;
  int T, K, V, v0, slab_w;
  float scale2;       // log2(e) / tau
};

// Plain fp32 output tile: store or accumulate.
struct F32Params {
  float* out;
  int64_t ldo;
  int M, N;
  int accumulate;
  int vec_ok;  // ldo and base allow 32-byte vector access
  // bf16 destination: when set, the tile (plus out's fp32 values when accumulating) is
  // rounded to bf16 and stored here instead of to out.
  uint16_t* out16 = nullptr;
  int64_t ldo16 = 0;
  int vec16_ok = 0;  // ldo16 and out16 allow 16-byte vector access
};

bool encode_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer);
// 3-D view of an MN-major operand stored [k][mn] (mn contiguous, mn_extent % 64 == 0 and
// every element below mn_extent inside the buffer): dims (64, k, mn_extent / 64), box
// (64, 64, tile_mn / 64).  Returns false if the map cannot be encoded.
bool encode_map_mn3d(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_extent,
                     uint64_t row_stride_bytes, uint32_t tile_mn);
// The same with 32-element atoms and the 64-byte swizzle (two-SM B halves 96 wide); the
// 2-D form loads one 32 x 64 box.  mn_extent % 32 == 0 for the 3-D form.
bool encode_map_mn3d_sw64(CUtensorMap* map, const void* base, uint64_t mn_extent, uint64_t k_extent,
                          uint64_t row_stride_bytes, uint32_t tile_mn);
bool encode_map_bf16_sw64(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_stride_bytes);

cudaError_t launch_gemm_fwd(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                            const FwdParams& ep, int grid, cudaStream_t st);
// Two-SM (CTA pair) versions: 256-row tiles; B maps load BN/2 rows (or columns) per CTA;
// the grid is sized from the clusters that fit on the device (sms = SM count).
cudaError_t launch_gemm2_fwd(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                             const FwdParams& ep, int sms, cudaStream_t st);
cudaError_t launch_gemm2_ds(const CUtensorMap& a, const CUtensorMap& b, const GemmShape& g,
                            const DsParams& ep, int sms, cudaStream_t st);
cudaError_t launch_gemm2_f32(int bn, bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmShape& g, const F32Params& ep, int sms, cudaStream_t st);
// Adds the K pieces of every split unit of `g` (plan_ksplit) in piece order into ep.out.
cudaError_t launch_ksplit_fixup(int bn, const GemmShape& g, const F32Params& ep, cudaStream_t st);
// F32-output GEMM for bn in {256, 192, 128} and either major-ness of A and B.
cudaError_t launch_gemm_f32(int bn, bool a_mn, bool b_mn, const CUtensorMap& a,
                            const CUtensorMap& b, const GemmShape& g, const F32Params& ep,
                            int grid, cudaStream_t st);

}  // namespace fkl
