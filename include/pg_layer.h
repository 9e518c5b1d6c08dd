/*
 * Building blocks of one Llama-style decoder layer run over packed shared-prefix groups: the
 * linear projections of the layer are applied to the packed tokens, so the shared prefix passes
 * through them once per group rather than once per response (abstract page of Prefix Grouper:
 * the shared prefix is encoded only once; Pith review, "Core claim": the cost ratio tends to 1/G).
 * Same conventions as pg_grouped_attn.h: caller-owned device buffers, asynchronous on `stream`,
 * host-side argument checks, no allocation.
 */
#ifndef PG_LAYER_H
#define PG_LAYER_H

#include "pg_grouped_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * C[m, n] = sum_k A(m, k) * B(n, k) on the tensor cores (bf16 inputs, fp32 accumulation).
 *   A(m, k) = A[m * lda + k] if a_mn == 0 (row-major [M, K]), A[k * lda + m] if a_mn == 1
 *   B(n, k) = B[n * ldb + k] if b_mn == 0 (row-major [N, K]), B[k * ldb + n] if b_mn == 1
 * C is row-major [M, ldc] of c_dtype (PG_F32 or PG_BF16), overwritten.  With a_mn = b_mn = 0 this
 * is X W^T of a linear layer; b_mn = 1 gives dY W (input gradient); a_mn = 1, b_mn = 1 gives
 * dY^T X (weight gradient).  Requirements: device pointers, A and B 16-byte aligned, lda and ldb
 * multiples of 8 covering their rows, ldc >= N.
 * Errors: PG_ERR_INVALID_ARG (host check, nothing launched); PG_ERR_CUDA on a launch failure.
 */
pg_status pg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int32_t a_mn, int64_t lda,
                       const void* B, int32_t b_mn, int64_t ldb, void* C, pg_dtype c_dtype,
                       int64_t ldc, pg_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PG_LAYER_H */
