/*
 * fkl_testing.h - test hooks of the fused chunked KL library.
 *
 * These entry points expose single building blocks of the loss so that each can be
 * checked on its own against a float64 host reference.  They are not part of the loss's
 * API and the pages have no counterpart for them.  Conventions (pointers, alignment,
 * streams, status codes) are those of fkl.h.
 */
#ifndef FKL_TESTING_H_
#define FKL_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#include "fkl.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * The tensor-core GEMM that the loss is built from, with a plain fp32 epilogue:
 *   D[M, N] (fp32, row-major, leading dimension N) = A B^T      if (accumulate & 1) == 0
 *   D[M, N] += A B^T                                             if (accumulate & 1) != 0
 * A is logically [M, Kd] and B logically [N, Kd], both bfloat16.  a_mn_major = 0 means A is
 * stored [M][Kd] (Kd contiguous); 1 means stored [Kd][M] (M contiguous).  Likewise for B.
 * bn selects the tile width along N: 256, 192 or 128.  M, N, Kd >= 1; the contiguous
 * extent of each operand must be a multiple of 8.  An MN-major operand whose extent is a
 * multiple of 64 is loaded with one 3-D TMA box per tile, unless bit 1 of `accumulate` is
 * set (then 64-wide 2-D boxes, the path used for other extents).  Bit 0 of `accumulate`
 * selects accumulation.  Bit 2 selects the two-SM kernel (CTA pairs, 256-row tiles, the one
 * the loss uses; a 192-wide tile with MN-major B uses the 64-byte swizzle) instead of the one-SM kernel (128-row tiles).  Bit 3
 * (with bit 2) splits the units of the last, partial wave of CTA pairs along K, as the
 * backward does for dW and dH: their partial tiles go to the workspace after the first 256
 * bytes (256 x bn fp32 each, as many as fit, at most 80) and a fixup kernel adds them.
 * `workspace` needs 256 bytes (the status word) and the partial tiles' room.
 */
fkl_status fkl_test_gemm(const uint16_t* A, const uint16_t* B, float* D, int64_t M, int64_t N,
                         int64_t Kd, int a_mn_major, int b_mn_major, int bn, int accumulate,
                         void* workspace, size_t ws_bytes, void* stream);

/*
 * The backward's blocking for this shape on a device with `sms` SMs (host only, no device
 * call): out[0] = tokens per block Ct, out[1] = token blocks, out[2] = vocabulary columns per
 * slab Vc, out[3] = vocabulary slabs, out[4] = the widest slab the workspace's dS buffer
 * holds (Ct x out[4] bf16 values; Vc <= out[4]).  out has room for 5 values.  Returns
 * FKL_ERR_INVALID_ARG for shapes fkl_workspace_size rejects or sms < 2.
 */
fkl_status fkl_test_backward_plan(int64_t T, int64_t d, int64_t V, int64_t K, int64_t chunk, int32_t sms,
                                  int64_t* out);

/*
 * Runs one pipeline wait on a barrier that nothing completes, with a time limit of
 * limit_ns nanoseconds (at most one second), so that the bounded-wait path can be
 * checked without hanging the GPU: afterwards fkl_read_status(workspace, stream) must
 * return FKL_ERR_TIMEOUT.  `workspace` needs 256 bytes.
 */
fkl_status fkl_test_wait_timeout(uint64_t limit_ns, void* workspace, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FKL_TESTING_H_ */
