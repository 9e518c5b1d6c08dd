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
 * C[m, n] (+)= sum_k A(m, k) * B(n, k) on the tensor cores (bf16 inputs, fp32 accumulation).
 *   A(m, k) = A[m * lda + k] if a_mn == 0 (row-major [M, K]), A[k * lda + m] if a_mn == 1
 *   B(n, k) = B[n * ldb + k] if b_mn == 0 (row-major [N, K]), B[k * ldb + n] if b_mn == 1
 * C is row-major [M, ldc] of c_dtype (PG_F32 or PG_BF16): overwritten when accumulate == 0,
 * C + A B^T (added in fp32, then stored) when accumulate == 1.  With a_mn = b_mn = 0 this is X W^T
 * of a linear layer; b_mn = 1 gives dY W (input gradient); a_mn = 1, b_mn = 1 gives dY^T X
 * (weight gradient).  Requirements: device pointers, A and B 16-byte aligned, lda and ldb
 * multiples of 8 covering their rows, ldc >= N.
 * Errors: PG_ERR_INVALID_ARG (host check, nothing launched); PG_ERR_CUDA on a launch failure.
 */
pg_status pg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int32_t a_mn, int64_t lda,
                       const void* B, int32_t b_mn, int64_t ldb, void* C, pg_dtype c_dtype,
                       int64_t ldc, int32_t accumulate, pg_stream_t stream);

/*
 * The q or k projection with RoPE in its epilogue: C[m, n] = rotate(sum_k A[m * lda + k] *
 * B[n * ldb + k]) in bf16, where every head_dim-wide column block of a row m is rotated as the
 * attention calls rotate q and k (rotate-half pairs (j, j + head_dim/2), j < head_dim/2, by the
 * angle whose (cos, sin) is table[m * head_dim/2 + j]): the fp32 accumulator is rotated before
 * the one rounding to bf16.  table: the float2 [table_rows][head_dim/2] table of pg_rope_table
 * (table_rows = the layout's total tokens, at least M; row m of A is token m).  A and B
 * row-major (K-major), bf16, 16-byte aligned, lda and ldb multiples of 8; C bf16, 16-byte
 * aligned, ldc a multiple of 8 and >= N; head_dim 64 or 128 dividing N.  The result feeds the
 * attention calls with PG_FLAG_PRE_ROTATED.
 * Errors: PG_ERR_INVALID_ARG (host check, nothing launched); PG_ERR_CUDA on a launch failure.
 */
pg_status pg_gemm_bf16_rope(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                            const void* B, int64_t ldb, void* C, int64_t ldc, int32_t head_dim,
                            const void* table, int64_t table_rows, pg_stream_t stream);

/*
 * RMSNorm forward over T rows of `hidden` bf16 values (Llama style: no mean subtraction):
 *   y = x + residual (stored to sum_out in bf16, when residual is not NULL), else y = x;
 *   out = y / sqrt(mean(y^2) + eps) * gamma  (bf16);  rstd[t] = 1 / sqrt(mean(y_t^2) + eps) (fp32).
 * x, residual, sum_out, out: [T, hidden] bf16; gamma: [hidden] bf16.  sum_out may alias neither
 * x nor residual.  Errors: PG_ERR_INVALID_ARG for bad sizes or pointers.
 */
pg_status pg_rmsnorm_fwd(int64_t T, int32_t hidden, const void* x, const void* residual,
                         const void* gamma, float eps, void* out, void* sum_out, float* rstd,
                         pg_stream_t stream);

/* Workspace bytes pg_rmsnorm_bwd needs for T rows of width hidden. */
size_t pg_rmsnorm_bwd_workspace(int64_t T, int32_t hidden);

/*
 * RMSNorm backward: with yhat = y * rstd,
 *   dx = dres + rstd * (gamma * dout - yhat * mean(yhat * gamma * dout))   (dres optional, bf16)
 *   dgamma = sum over rows of dout * yhat   (fp32 [hidden], summed in a fixed order)
 * y is the forward's normalised input (sum_out, or x), rstd its fp32 rows; dout and dx are
 * [T, hidden] in the stated dtypes.  workspace: device, >= pg_rmsnorm_bwd_workspace(T, hidden).
 */
pg_status pg_rmsnorm_bwd(int64_t T, int32_t hidden, const void* y, const void* gamma,
                         const float* rstd, const void* dout, pg_dtype dout_dtype,
                         const void* dres, void* dx, pg_dtype dx_dtype, float* dgamma,
                         void* workspace, size_t workspace_bytes, pg_stream_t stream);

/*
 * SwiGLU: gate_up is [T, 2 * inter] bf16 (gate columns first, then up); out[t, i] =
 * silu(gate[t, i]) * up[t, i], silu(g) = g / (1 + exp(-g)), bf16 [T, inter].
 */
pg_status pg_swiglu_fwd(int64_t T, int32_t inter, const void* gate_up, void* out,
                        pg_stream_t stream);

/* SwiGLU backward: dgate_up [T, 2 * inter] bf16 from gate_up and dout [T, inter]. */
pg_status pg_swiglu_bwd(int64_t T, int32_t inter, const void* gate_up, const void* dout,
                        void* dgate_up, pg_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* PG_LAYER_H */
