/*
 * fkl.h - C ABI of the fused chunked KL distillation loss for GB300 (sm_103a).
 *
 * The operation is the loss of "Efficient Knowledge Distillation for LLMs: Offline Top-K
 * Logits and a Fused Chunked KL Loss" (Hugging Face blog post, section "Two systems
 * changes", paragraphs "Offline distillation" and "Fused chunked KL"): the student's
 * final hidden states H are projected through the LM head W chunk by chunk, each chunk of
 * logits is folded into a running loss against the teacher's cached top-K logits and then
 * discarded, and the backward pass recomputes each chunk instead of storing it.  The
 * pages print no formula; the one implemented is
 *
 *     s = H W^T (bf16 inputs, fp32 accumulation),  a = s / tau
 *     lse_t = log sum_v exp(a_tv)                   over the whole vocabulary
 *     p_t   = softmax(z_t / tau)                    over the K cached teacher slots
 *     KL_t  = sum_k p_tk (log p_tk - (a_{t,id_tk} - lse_t))
 *     L     = tau^2 / N * sum_{t : mask_t = 1} KL_t,     N = number of valid tokens
 *
 * and its gradient (the post's "closed-form gradient", not printed there)
 *
 *     dS_tv = g * tau / N * (exp(a_tv - lse_t) - ptilde_tv)  for valid t, else 0
 *     dH = dS W,  dW = dS^T H                                  (fp32 outputs)
 *
 * where ptilde_t is p_t added at the ids of row t and g the upstream gradient of L.
 * N = 0 gives L = 0 and zero gradients.  No T x V tensor is ever written to memory:
 * logits live only in tensor memory, one tile at a time; the backward writes dS one block
 * (a range of tokens x a vocabulary slab) at a time into the caller's workspace, bounded
 * by `chunk` (below).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device memory of the current device (or managed memory);
 *     all buffers are row-major and contiguous.  A pointer that is not (host memory given
 *     by mistake) is refused on the host with FKL_ERR_INVALID_ARG before anything is
 *     enqueued.  The caller owns every buffer, including the workspace; the library
 *     allocates no device memory.
 *   - H and W are bfloat16 bit patterns (uint16_t).  H, W, dH and dW must be 16-byte
 *     aligned, the workspace 256-byte aligned, everything else 4-byte aligned; d must be a
 *     multiple of 8 (TMA rows are whole 16-byte units).  dH and dW are written with 32-byte
 *     vectors when they are 32-byte aligned (any CUDA allocation is) and element by element,
 *     more slowly, when they are not.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous
 *     on `stream`; they never synchronise the device.
 *   - Shape limits: 0 <= T < 2^31, 1 <= V < 2^31, 8 <= d < 2^20, d % 8 == 0,
 *     1 <= K <= 1024, chunk >= 1, tau > 0 and finite.
 *   - Errors found on the host (bad argument, alignment, workspace too small, a CUDA
 *     launch failure) are returned at once and nothing is enqueued after the failing
 *     step; fkl_last_error() gives a message.  Errors found on the device (a teacher id
 *     outside [0, V), a teacher row with no finite logit, a sequence id out of range, a
 *     pipeline wait that exceeded its time limit) are recorded in a status word inside the
 *     workspace, make the loss NaN (forward) or fill dH and dW with NaN (backward), and are
 *     reported by fkl_read_status().  No device code traps.
 *   - Results are deterministic: the same inputs give bitwise the same outputs.
 */
#ifndef FKL_H_
#define FKL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fkl_status {
  FKL_OK = 0,
  FKL_ERR_INVALID_ARG = 1,  /* NULL or non-device pointer, bad shape, non-positive tau or chunk */
  FKL_ERR_ALIGNMENT = 2,    /* a pointer or d breaks the alignment rules above */
  FKL_ERR_UNSUPPORTED = 3,  /* the current device is not sm_103 */
  FKL_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than fkl_workspace_size() */
  FKL_ERR_CUDA = 5,         /* a CUDA runtime or driver call failed */
  FKL_ERR_BAD_TOPK_ID = 6,  /* device: a teacher id is outside [0, V) */
  FKL_ERR_BAD_TOPK_ROW = 7, /* device: a teacher row has no finite logit */
  FKL_ERR_TIMEOUT = 8,      /* device: a pipeline wait exceeded its time limit */
  FKL_ERR_BAD_SEQ_ID = 9,   /* device: a valid token's sequence id is outside [0, num_seqs) */
  FKL_ERR_TOPK_OVERFLOW = 10, /* device: fkl_teacher_topk found more tied candidates than it holds */
  FKL_ERR_BAD_COUNT = 11      /* device: fkl_options.global_count is below this call's own count */
} fkl_status;

/*
 * Options of fkl_forward_ex / fkl_backward_ex (fkl_forward / fkl_backward use the defaults:
 * all fields zero).
 *
 * normalization  FKL_NORM_TOKENS (0): L = tau^2 / N * sum over valid tokens of KL_t, the
 *                mean over the batch's valid tokens.
 *                FKL_NORM_SEQUENCES (1): for packed batches, the mean over sequences of each
 *                sequence's token mean, L = tau^2 / S * sum_s (1 / N_s) sum_{valid t in s} KL_t,
 *                over the S sequences that have a valid token (N_s of them in sequence s).
 *                The pages mention sequence packing without fixing the normaliser; both
 *                readings are offered, the token mean is the default.
 * seq_ids        FKL_NORM_SEQUENCES: device int32 [T], the packed sequence of each token, in
 *                [0, num_seqs); any order.  Ignored otherwise (may be NULL).
 * num_seqs       FKL_NORM_SEQUENCES: 1 <= num_seqs <= max(T, 1).
 * accumulate     fkl_backward_ex: FKL_ACCUMULATE_DH and/or FKL_ACCUMULATE_DW add the gradient
 *                into dH / dW (gradient accumulation over micro-batches) instead of
 *                overwriting them.  Ignored by the forward.
 * divergence     The divergence D_t in place of KL_t (the post's closing section says the
 *                paper also compares loss functions without naming them).  With p the
 *                teacher's K-slot softmax added onto the vocabulary at its ids (zero at
 *                every other id; a repeated id carries the sum of its slots) and q_t the
 *                student's full softmax of s_t / tau:
 *                  FKL_DIV_KL (0)        KL(p || q), the loss above (default; a repeated id
 *                                        counts once per slot, as in KL_t's slot sum)
 *                  FKL_DIV_JSD (1)       b KL(p || m) + (1 - b) KL(q || m), m = b p + (1 - b) q,
 *                                        0 < b < 1 (b = 1/2: Jensen-Shannon)
 *                  FKL_DIV_SKEW_KL (2)   KL(p || a p + (1 - a) q), 0 <= a < 1
 *                  FKL_DIV_SKEW_RKL (3)  KL(q || a q + (1 - a) p), 0 < a <= 1
 *                  FKL_DIV_TV (4)        1/2 sum_v |p - q| (sign(0) = 0 in its gradient)
 *                all summed over the whole vocabulary, and L = tau^2 sum_t w_t D_t with the
 *                token weights w_t of `normalization`.  Each is finite where p is zero, so
 *                the K cached slots suffice: D_t = sum over the row's ids of a term in
 *                (p, q) plus a constant times the student mass outside them.
 * div_param      b for FKL_DIV_JSD, a for FKL_DIV_SKEW_KL / FKL_DIV_SKEW_RKL; ignored
 *                otherwise.
 * student_topk_logits
 *                device float [T, K] or NULL.  fkl_forward_ex writes s_{t, id_tk}, the
 *                student's logit (fp32, before 1/tau) at each cached slot, when it is not
 *                NULL.  fkl_backward_ex reads it for every divergence but FKL_DIV_KL (the
 *                gradient needs q at the ids before the vocabulary sweep), so it must then
 *                hold the forward's values for the same inputs; it is ignored for KL.
 * global_count   device int64 scalar, or NULL (the default: the call's own count).  The count
 *                that the mean divides by, taken over the whole batch when the batch is split
 *                over several calls: token shards on data-parallel ranks, or the micro-batches
 *                of one accumulated step.  It is the number of valid tokens of the whole batch
 *                (FKL_NORM_TOKENS), or the number of its sequences with a valid token
 *                (FKL_NORM_SEQUENCES; each sequence must then lie within one call, which is
 *                how packed sequences are sharded).  The token weights become
 *                w_t = 1 / global_count or 1 / (global_count * N_s), so the calls' losses add
 *                up to the batch's loss and their dH rows and summed dW are the batch's
 *                gradient.  Sum fkl_local_count over the calls (an all-reduce on the device
 *                across ranks) to get it; it is read on the device, so no host round trip is
 *                needed.  If it is below the call's own count the device records
 *                FKL_ERR_BAD_COUNT (loss NaN, gradients NaN).  8-byte aligned.  The forward
 *                and the backward of one step must be given the same value.
 */
enum { FKL_NORM_TOKENS = 0, FKL_NORM_SEQUENCES = 1 };
enum { FKL_ACCUMULATE_DH = 1, FKL_ACCUMULATE_DW = 2 };
enum { FKL_DIV_KL = 0, FKL_DIV_JSD = 1, FKL_DIV_SKEW_KL = 2, FKL_DIV_SKEW_RKL = 3, FKL_DIV_TV = 4 };
typedef struct fkl_options {
  int32_t normalization;
  int32_t num_seqs;
  const int32_t* seq_ids;
  int32_t accumulate;
  int32_t divergence;
  float div_param;
  int32_t reserved;  /* must be 0 */
  float* student_topk_logits;
  const int64_t* global_count;
} fkl_options;

/*
 * This call's own count, the term of fkl_options.global_count that this shard contributes:
 * writes to *count (device int64) the number of valid tokens (FKL_NORM_TOKENS, opts NULL or
 * opts->normalization = 0), or the number of sequences with a valid token
 * (FKL_NORM_SEQUENCES, from opts->seq_ids / num_seqs).  Summed over the shards of a batch
 * (with an all-reduce of the device scalar across data-parallel ranks, or a device add over
 * micro-batches) it gives the batch's global_count.  The pages' GPT-OSS 20B run trains on
 * one node of several GPUs and reports per-GPU throughput (the post's "Scaling to long
 * context lengths"); they do not say how its loss is normalised across GPUs.  The plainest
 * reading, taken here, is the loss of the whole batch: every shard divides by the batch's
 * count, not its own.
 *   mask       uint8 [T], 1 = valid; NULL = all valid
 *   workspace  device buffer of at least 256 + 4 * max(T, 1) bytes, 256-byte aligned (a
 *              workspace of fkl_workspace_size for the same T is large enough); a sequence
 *              id out of range is recorded in it for fkl_read_status (FKL_ERR_BAD_SEQ_ID)
 * Asynchronous on `stream`; 0 <= T < 2^31.
 */
fkl_status fkl_local_count(const uint8_t* mask, int64_t T, const fkl_options* opts, int64_t* count,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of workspace that fkl_forward and fkl_backward need for this shape (one buffer
 * serves both; no state is carried between calls in it).  `chunk` bounds the backward's
 * dS buffer: it holds one block of the backward (a range of tokens x a vocabulary slab of
 * whole 256-column tiles, at least one tile wide), at most chunk * V bfloat16 values.  The result
 * does not depend on `chunk` beyond floating-point summation order.  For T > 0 it also holds
 * 80 fp32 partial tiles of 256 x 256 (20 MiB) for the dW and dH units that the backward splits
 * along the reduction.  Returns 0 for invalid shapes.
 */
size_t fkl_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk);

/*
 * Number of blocks (token block x vocabulary slab) the backward pass walks for this shape
 * on the current device (the slab width depends on its SM count; a GB300's 152 SMs are
 * assumed when no device is visible): each is one dS-recompute GEMM, one dW GEMM and one dH
 * GEMM launch.  0 for T = 0 or invalid shapes.
 */
int64_t fkl_backward_slabs(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk);

/*
 * Forward pass: writes the scalar loss L to *loss (device float) and lse[t] (device
 * float[T], natural log of sum_v exp(s_tv / tau), defined for masked tokens too).
 *   H           bf16 [T, d]     student final hidden states
 *   W           bf16 [V, d]     LM-head weight
 *   topk_idx    int32 [T, K]    teacher's cached top-K token ids, any slot order
 *   topk_logits fp32 [T, K]     teacher's logits for those ids (-inf allowed per slot)
 *   mask        uint8 [T]       1 = token counts, 0 = skipped; NULL = all tokens count
 *   workspace   device buffer of ws_bytes >= fkl_workspace_size(T, d, V, K, chunk)
 */
fkl_status fkl_forward(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                       const float* topk_logits, const uint8_t* mask, int64_t T, int64_t d,
                       int64_t V, int64_t K, float tau, int64_t chunk, float* loss, float* lse,
                       void* workspace, size_t ws_bytes, void* stream);

/* fkl_forward with options (NULL = defaults). */
fkl_status fkl_forward_ex(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                          const float* topk_logits, const uint8_t* mask, int64_t T, int64_t d,
                          int64_t V, int64_t K, float tau, int64_t chunk, const fkl_options* opts,
                          float* loss, float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward pass: recomputes the projection chunk by chunk and writes dH (device float
 * [T, d]) and dW (device float [V, d]); both are overwritten, not accumulated into.
 *   lse        device float [T] from fkl_forward on the same inputs
 *   grad_loss  device float scalar g (the upstream gradient of L); NULL means g = 1
 * Other arguments as in fkl_forward.
 */
fkl_status fkl_backward(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                        const float* topk_logits, const uint8_t* mask, const float* lse,
                        const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K,
                        float tau, int64_t chunk, float* dH, float* dW, void* workspace,
                        size_t ws_bytes, void* stream);

/*
 * Forward pass for callers that cannot allocate device memory - for example a custom
 * operator inside another runtime that owns the whole device memory pool and passes the op
 * only its input and output tensors, or a latency-critical loop that must never call
 * cudaMalloc.  The pages have no counterpart for this entry point: it is a packaging
 * option of this library, not part of the method.
 *
 * Same arguments as fkl_forward, without `chunk` (the forward does not depend on it) and
 * without a workspace: the scratch lives in a 64 MiB device array inside the library, which
 * every GPU that loads the library keeps until the process exits.  Shapes whose forward
 * scratch exceeds it (about T * (8K + 400) bytes; T up to about 56K tokens at K = 100) are
 * rejected with FKL_ERR_WORKSPACE and a message in fkl_last_error().
 *   - The results equal fkl_forward's within the parity tolerances (loss relative 1e-3, lse
 *     absolute 1e-3) but not bit for bit: this path runs the one-SM GEMM, whose vocabulary
 *     splits differ from the two-SM forward's, so the fp32 partial sums merge in another
 *     order.  Repeated calls on the same inputs give bitwise the same outputs.
 *   - The first call on a device sets it up (loads the library's module there, checks the
 *     device and reads its SM count); make that first call before any stream capture.
 *     Every call looks up the array's device address with the device current.
 *   - All calls share the one array and it keeps the last call's contents (each call
 *     clears what must start at zero): calls that overlap on the GPU - on different
 *     streams or from different threads - race and must be serialised by the caller.
 *   - It allocates nothing (no cudaMalloc or allocating library routine).  A device-side
 *     error (bad teacher id or row, pipeline timeout) makes the loss NaN; its status word
 *     is internal and cannot be read with fkl_read_status.
 */
fkl_status fkl_forward_noalloc(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                               const float* topk_logits, const uint8_t* mask, int64_t T,
                               int64_t d, int64_t V, int64_t K, float tau, float* loss, float* lse,
                               void* stream);

/* fkl_backward with options (NULL = defaults).  With the same options as the forward. */
fkl_status fkl_backward_ex(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                           const float* topk_logits, const uint8_t* mask, const float* lse,
                           const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K,
                           float tau, int64_t chunk, const fkl_options* opts, float* dH, float* dW,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Backward pass with bfloat16 gradients: the same computation as fkl_backward_ex, with dH
 * [T, d] and dW [V, d] written as bfloat16 (uint16_t bit patterns, rounded to nearest even)
 * instead of float.  The sums stay fp32 until their last term: dH of a token block is summed
 * over the vocabulary slabs in an fp32 buffer in the workspace and rounded when the last
 * slab is added; dW is rounded when its last token block is added (with several token
 * blocks its sums live in an fp32 [V, d] buffer in the workspace).  The result equals
 * fkl_backward_ex's fp32 result rounded to bfloat16, bit for bit.  The bf16 outputs halve
 * the gradients' memory (dW is 1.16 GB instead of 2.32 GB at V = 201088, d = 2880) and are
 * what a bf16 model's autograd wants.  opts->accumulate must be 0 (FKL_ERR_INVALID_ARG
 * otherwise); dH and dW must be 16-byte aligned.  The workspace must hold
 * fkl_backward_bf16_workspace_size bytes (it serves fkl_forward as well).
 */
fkl_status fkl_backward_bf16(const uint16_t* H, const uint16_t* W, const int32_t* topk_idx,
                             const float* topk_logits, const uint8_t* mask, const float* lse,
                             const float* grad_loss, int64_t T, int64_t d, int64_t V, int64_t K, float tau,
                             int64_t chunk, const fkl_options* opts, uint16_t* dH, uint16_t* dW,
                             void* workspace, size_t ws_bytes, void* stream);

/* Bytes of workspace fkl_backward_bf16 needs: fkl_workspace_size plus the fp32 sums (Ct x d
 * floats for dH's token block; V x d more when the backward takes several token blocks).
 * 0 for invalid shapes. */
size_t fkl_backward_bf16_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk);

/*
 * Waits for `stream`, then returns the device-side status recorded in `workspace` by the
 * most recent fkl_forward / fkl_backward call that used it (FKL_OK if none failed), or
 * FKL_ERR_CUDA if the wait or the read fails.
 */
fkl_status fkl_read_status(const void* workspace, void* stream);

/*
 * Per-launch timing for profiling.  After fkl_trace_start(capacity) the calling thread's
 * fkl_forward and fkl_backward calls record a CUDA event pair on the caller's stream around
 * each of their tensor-core GEMM launches, for the first `capacity` launches (1..65536);
 * fkl_trace_stop() ends recording.  The events are created by the library when the trace
 * starts (no device memory is allocated) and are released by the next fkl_trace_start.
 */
fkl_status fkl_trace_start(int32_t capacity);
fkl_status fkl_trace_stop(void);

/*
 * Waits for the recorded events and writes, for up to `capacity` recorded launches in launch
 * order, the duration in milliseconds (ms), the kind (0 forward projection + logsumexp,
 * 1 dS recompute, 2 dW, 3 dH, 4 the fixup that completes the K-split units of the dW or dH
 * launch recorded just before it, with 0 FLOPs, 5 teacher top-K bound pass, 6 teacher top-K
 * candidate pass)
 * and the launch's algorithmic FLOPs (2 * M * N * K of its product).  Any output pointer may be NULL.  Returns the number written, -1 on a CUDA error.
 */
int32_t fkl_trace_read(float* ms, int32_t* kind, double* flops, int32_t capacity);

/*
 * Offline teacher cache ("Two systems changes", paragraph "Offline distillation": the teacher
 * runs once and the top-100 tokens per position are stored): for the teacher's final hidden
 * states Ht (bf16 [T, d]) and LM head Wt (bf16 [V, d]), writes the K largest logits of each
 * row of s = Ht Wt^T (fp32 accumulation) and their ids, ordered by logit descending, ties by
 * the lower id: topk_idx int32 [T, K] and topk_logits fp32 [T, K] - the cache that
 * fkl_forward reads.  The T x V logits are never written.  A first pass over every s-th
 * vocabulary row (s = 8 for large V; fewer when V is small) finds a per-row lower bound of
 * the K-th largest logit; a second, full projection collects the logits at or above it (at
 * most max(512, 4 s K) per row; more, which needs massive ties or a teacher whose largest
 * logits all avoid the sampled rows, is reported as FKL_ERR_TOPK_OVERFLOW with id -1 and
 * logit NaN in that row).  The result is exact either way.  Limits: 1 <= K <= V,
 * d % 8 == 0; when V > 4096 also K <= 256 and K <= 8 * ceil(V / 256).
 */
size_t fkl_teacher_topk_workspace_size(int64_t T, int64_t d, int64_t V, int64_t K);
fkl_status fkl_teacher_topk(const uint16_t* Ht, const uint16_t* Wt, int64_t T, int64_t d, int64_t V,
                            int64_t K, int32_t* topk_idx, float* topk_logits, void* workspace,
                            size_t ws_bytes, void* stream);

/*
 * fkl_teacher_topk with a cap on the bound pass's sampling stride: max_bound_stride = 1 reads
 * every vocabulary row in the first pass (its bound is then the K-th largest of every split's
 * largest logits, the tightest one, and the second pass collects at most about 4K per row),
 * 2, 4 or 8 allow sampling, 0 is the default (8).  A run that reported FKL_ERR_TOPK_OVERFLOW
 * because of sampling succeeds with 1.  The workspace of fkl_teacher_topk_workspace_size
 * serves every stride.  Other errors as fkl_teacher_topk, plus FKL_ERR_INVALID_ARG for
 * another max_bound_stride.
 */
fkl_status fkl_teacher_topk_ex(const uint16_t* Ht, const uint16_t* Wt, int64_t T, int64_t d, int64_t V,
                               int64_t K, int32_t max_bound_stride, int32_t* topk_idx, float* topk_logits,
                               void* workspace, size_t ws_bytes, void* stream);

/* Static text for a status code. */
const char* fkl_status_string(int status);

/* Message of the last host-side error on the calling thread ("" if none). */
const char* fkl_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FKL_H_ */
