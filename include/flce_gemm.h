/*
 * flce_gemm.h - the raw tensor-core contraction under the fused linear
 * cross-entropy, exported on its own so that its operand layouts can be
 * checked in isolation.
 *
 * It is the contraction of Liger-Kernel issue #533 "Gradient checkpointing for
 * grad_weight in LFCE" (feature pitch: grad_weight accumulated by an addmm with
 * beta = 1 and alpha = 1), generalised to every operand layout the loss head
 * needs:
 *
 *     C[m, n] (+)= sum_k A[m, k] * B[n, k]        (fp32 accumulation, fp32 C)
 *
 * A is K-major (a_mn_major = 0: row m at A + m*lda, K contiguous) or MN-major
 * (a_mn_major = 1: row k at A + k*lda, M contiguous); likewise B.  Inputs are
 * bf16 (FLCE_BF16, tcgen05 kind::f16) or fp32 (FLCE_F32, tcgen05 kind::tf32).
 * The tf32 tensor-core path reads K-major operands only: FLCE_F32 with either
 * operand MN-major returns FLCE_ENOSUP.
 * accumulate = 1 adds to the existing C (beta = 1), 0 overwrites it.
 *
 * All pointers are device pointers, 16-byte aligned; lda*sizeof(dt) and
 * ldb*sizeof(dt) must be multiples of 16 and ldc a multiple of 4.  The call is
 * enqueued on `stream`, allocates nothing and never synchronises.  Errors are
 * reported as in flce.h (a timed-out wait inside the kernel writes
 * FLCE_ETIMEOUT to *status).
 */
#ifndef FLCE_GEMM_H
#define FLCE_GEMM_H

#include "flce.h"

#ifdef __cplusplus
extern "C" {
#endif

FLCE_API int flce_gemm(int dt, int a_mn_major, int b_mn_major, int64_t M, int64_t N, int64_t K,
              const void* A, int64_t lda, const void* B, int64_t ldb, float* C, int64_t ldc,
              int accumulate, int32_t* status, flce_stream_t stream);

/* Selects how each bf16 contraction is tiled.  `mask` has one bit per
 * contraction: 1 the forward logits, 2 the backward recompute of dZ, 4 grad_H,
 * 8 grad_W, 16 flce_gemm itself.  A set bit runs each 256 x 256 tile on a pair
 * of CTAs on two SMs (tcgen05.mma.cta_group::2, each SM loading half of B); a
 * clear bit runs each 128 x 256 tile on one CTA.  Both give the same results up
 * to fp32 summation order.  Bit 32 is not a contraction: when set, the dZ
 * recompute at K = D <= 1024 runs on one CTA per tile with eight epilogue
 * warps instead (two per TMEM lane quarter, each forming half of the tile's
 * columns), whatever bit 2 says.  The default (2 | 8 | 16 | 32) is the faster
 * choice per contraction measured on GB300.  Returns the previous mask.  Process-wide; do
 * not change it while calls run. */
FLCE_API int flce_gemm_set_pair(int mask);

/* How many CTA pairs of the pair-tiled contraction can be resident at once on
 * the current device (SMs pair up within a GPC), or -1 on error. */
FLCE_API int flce_gemm_pair_slots(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_GEMM_H */
