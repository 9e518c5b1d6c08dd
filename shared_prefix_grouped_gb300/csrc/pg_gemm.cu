// BF16 GEMM on the 5th-generation tensor cores: TMA-staged operands (128-byte swizzle), tcgen05.mma
// issued by one thread, fp32 accumulator in TMEM, read back with tcgen05.ld for the epilogue.
//
//   C[m, n] = sum_k A(m, k) * B(n, k)
//   A(m, k) = A[m * lda + k] (K-major)  or  A[k * lda + m] (MN-major, "transposed")
//   B(n, k) = B[n * ldb + k] (K-major)  or  B[k * ldb + n] (MN-major)
//
// One CTA computes a 128 x 256 tile of C; 4 warps: warp 0 issues TMA loads into a 4-stage ring,
// warp 1 issues the MMAs (128 x 256 x 16 each, 4 per 64-wide K block, descriptors built once and
// advanced by constant offsets), then all four warps drain TMEM (warp w owns accumulator lanes /
// C rows 32w .. 32w + 31) with 16-byte stores where the tile is in bounds and aligned.
//
// The RoPE variant (the q / k projections feeding the attention calls with PG_FLAG_PRE_ROTATED)
// rotates every head_dim-wide column block of the accumulator in its epilogue: a thread holds a
// whole row, so each rotate-half pair (j, j + head_dim/2) is read from TMEM by the same thread,
// rotated in fp32 by its row's (cos, sin) from the table and rounded to bf16 once.  A 256-wide
// tile starts on a head boundary (head_dim 64 or 128 divides 256), so no pair straddles tiles.
#include "pg_internal.h"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int GROUP_M = 16;
constexpr uint32_t A_BYTES = BM * BK * 2;      // 16 KiB per stage
constexpr uint32_t B_BYTES = BN * BK * 2;      // 32 KiB per stage
constexpr uint64_t WAIT_NS = 2000000000ull;    // 2 s bound on every wait

__device__ int s_status_gemm = 0;

struct GemmSmem {
  uint8_t a[STAGES][A_BYTES];
  uint8_t b[STAGES][B_BYTES];
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t done;
  uint32_t tmem;
};

template <int A_MN, int B_MN, typename OutT, bool ROPE>
__global__ void __launch_bounds__(128, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                 OutT* __restrict__ C, int M, int N, int K, long long ldc, int accumulate,
                 int vec_ok, const float2* __restrict__ rope_tab, int head_dim) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  GemmSmem& sm = *reinterpret_cast<GemmSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Grouped rasterisation: consecutive CTAs walk down GROUP_M row blocks before moving to the
  // next column block, so a wave of CTAs touches a compact block of A rows and B columns that
  // stays in L2.
  const int num_m = (M + BM - 1) / BM, num_n = (N + BN - 1) / BN;
  const int tile = blockIdx.x;
  const int group = tile / (GROUP_M * num_n);
  const int first_m = group * GROUP_M;
  const int gm = min(num_m - first_m, GROUP_M);
  const int in_group = tile - group * GROUP_M * num_n;
  const int m0 = (first_m + in_group % gm) * BM, n0 = (in_group / gm) * BN;
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sm.tmem, BN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  bool ok = true;
  int issued = 0;   // TMA stages issued by the producer

  if (warp == 0) {
    if (elect_one()) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tb);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (!mbar_wait(&sm.empty[s], ph ^ 1, WAIT_NS)) { ok = false; break; }
        mbar_expect_tx(&sm.full[s], A_BYTES + B_BYTES);
        if (!A_MN) {
          tma_load_2d(sm.a[s], &ta, &sm.full[s], kb * BK, m0);
        } else {
          tma_load_2d(sm.a[s], &ta, &sm.full[s], m0, kb * BK);
          tma_load_2d(sm.a[s] + A_BYTES / 2, &ta, &sm.full[s], m0 + 64, kb * BK);
        }
        if (!B_MN) {
          tma_load_2d(sm.b[s], &tb, &sm.full[s], kb * BK, n0);
        } else {
#pragma unroll
          for (int q4 = 0; q4 < BN / 64; ++q4)
            tma_load_2d(sm.b[s] + q4 * (BK * 64 * 2), &tb, &sm.full[s], n0 + 64 * q4, kb * BK);
        }
        ++issued;
      }
      // Do not leave the kernel with copies in flight: wait (bounded) for the last stages.
      for (int kb = (issued > STAGES ? issued - STAGES : 0); kb < issued; ++kb)
        mbar_wait(&sm.full[kb % STAGES], (kb / STAGES) & 1, WAIT_NS);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, A_MN, B_MN);
      // MN-major: the next 64-wide M/N block is LBO further (the next TMA box).
      const uint64_t ad0 = A_MN ? sdesc_sw128(smem_u32(sm.a[0]), A_BYTES / 2, 1024)
                                : sdesc_sw128(smem_u32(sm.a[0]), 16, 1024);
      const uint64_t bd0 = B_MN ? sdesc_sw128(smem_u32(sm.b[0]), BK * 64 * 2, 1024)
                                : sdesc_sw128(smem_u32(sm.b[0]), 16, 1024);
      for (int kb = 0; kb < nk; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&sm.full[s], (kb / STAGES) & 1, WAIT_NS)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = desc_add(ad0, s * A_BYTES), bd = desc_add(bd0, s * B_BYTES);
        const uint32_t acc0 = kb != 0;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss(tmem, desc_add(ad, A_MN ? kk * 2048 : kk * 32),
                 desc_add(bd, B_MN ? kk * 2048 : kk * 32), idesc, kk == 0 ? acc0 : 1u);
        mma_commit(&sm.empty[s]);
      }
      mma_commit(&sm.done);
    }
    __syncwarp();
  }

  // Epilogue: every warp drains its 32 accumulator lanes.
  if (!mbar_wait(&sm.done, 0, WAIT_NS)) ok = false;
  ok = __all_sync(0xffffffffu, ok);     // the TMEM loads below are warp-collective
  tc_fence_after();
  const int row = m0 + warp * 32 + lane;
  if constexpr (ROPE) {
    // bf16 output, 16-byte stores (checked on the host), whole heads (head_dim divides N).
    const int half = head_dim >> 1;
    const float4* tab =
        reinterpret_cast<const float4*>(rope_tab + (size_t)(row < M ? row : M - 1) * half);
#pragma unroll 1
    for (int hc = 0; ok && hc < BN; hc += head_dim) {
#pragma unroll 1
      for (int j0 = 0; j0 < half; j0 += 32) {
        uint32_t x1[32], x2[32];
        const uint32_t t = tmem + ((uint32_t)(warp * 32) << 16) + hc + j0;
        tmem_ld32(t, x1);
        tmem_ld32(t + half, x2);
        tmem_ld_wait();
        if (row < M && n0 + hc < N) {
          float lo[32], hi[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float4 e = tab[(j0 + j) >> 1];      // (cos, sin) of pairs j0 + j, j0 + j + 1
            const float a0 = __uint_as_float(x1[j]), b0 = __uint_as_float(x2[j]);
            const float a1 = __uint_as_float(x1[j + 1]), b1 = __uint_as_float(x2[j + 1]);
            lo[j] = a0 * e.x - b0 * e.y;
            hi[j] = b0 * e.x + a0 * e.y;
            lo[j + 1] = a1 * e.z - b1 * e.w;
            hi[j + 1] = b1 * e.z + a1 * e.w;
          }
          OutT* dst = C + (long long)row * ldc + n0 + hc + j0;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 w;
            w.x = pack_bf16x2(lo[j], lo[j + 1]);
            w.y = pack_bf16x2(lo[j + 2], lo[j + 3]);
            w.z = pack_bf16x2(lo[j + 4], lo[j + 5]);
            w.w = pack_bf16x2(lo[j + 6], lo[j + 7]);
            *reinterpret_cast<uint4*>(dst + j) = w;
            w.x = pack_bf16x2(hi[j], hi[j + 1]);
            w.y = pack_bf16x2(hi[j + 2], hi[j + 3]);
            w.z = pack_bf16x2(hi[j + 4], hi[j + 5]);
            w.w = pack_bf16x2(hi[j + 6], hi[j + 7]);
            *reinterpret_cast<uint4*>(dst + half + j) = w;
          }
        }
      }
    }
  } else if (ok) {
    // 16-byte stores need the row start aligned: ldc * sizeof(OutT) a multiple of 16 and an
    // aligned C (checked on the host: vec_ok).
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, r);
      tmem_ld_wait();
      const int col0 = n0 + c * 32;
      if (row < M && col0 < N) {
        OutT* dst = C + (long long)row * ldc + col0;
        if (vec_ok && col0 + 32 <= N) {
          if constexpr (sizeof(OutT) == 4) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 v = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                     __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
              if (accumulate) {
                const float4 o = *reinterpret_cast<const float4*>(dst + j);
                v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
              }
              *reinterpret_cast<float4*>(dst + j) = v;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r[j + e]);
              if (accumulate) {
                const uint4 o = *reinterpret_cast<const uint4*>(dst + j);
                const __nv_bfloat16* ob = reinterpret_cast<const __nv_bfloat16*>(&o);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] += __bfloat162float(ob[e]);
              }
              uint4 w;
              w.x = pack_bf16x2(f[0], f[1]);
              w.y = pack_bf16x2(f[2], f[3]);
              w.z = pack_bf16x2(f[4], f[5]);
              w.w = pack_bf16x2(f[6], f[7]);
              *reinterpret_cast<uint4*>(dst + j) = w;
            }
          }
        } else {
          for (int j = 0; j < 32; ++j) {
            if (col0 + j < N) {
              float x = __uint_as_float(r[j]);
              if (accumulate) x += (float)dst[j];
              if constexpr (sizeof(OutT) == 4) dst[j] = x;
              else dst[j] = __float2bfloat16_rn(x);
            }
          }
        }
      }
    }
  }
  if (!ok) atomicCAS(&s_status_gemm, 0, (int)PG_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, BN);
  }
}

template <int A_MN, int B_MN, typename OutT, bool ROPE = false>
pg_status launch(const CUtensorMap& ta, const CUtensorMap& tb, void* C, int M, int N, int K,
                 long long ldc, int acc, cudaStream_t s, const float2* rope_tab = nullptr,
                 int head_dim = 0) {
  auto kern = gemm_bf16_kernel<A_MN, B_MN, OutT, ROPE>;
  const size_t smem = sizeof(GemmSmem) + 1024;
  pg_status st = cuda_check(
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
      "gemm smem attribute");
  if (st != PG_OK) return st;
  dim3 grid((unsigned)(((N + BN - 1) / BN) * ((M + BM - 1) / BM)));
  prof_begin(PG_KERNEL_GEMM, s);
  const int vec_ok = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) &&
                     ((ldc * (long long)sizeof(OutT)) % 16 == 0);
  kern<<<grid, 128, smem, s>>>(ta, tb, static_cast<OutT*>(C), M, N, K, ldc, acc, vec_ok,
                               rope_tab, head_dim);
  prof_end(PG_KERNEL_GEMM, s);
  return cuda_check(cudaGetLastError(), "gemm launch");
}

}  // namespace

pg_status read_status_gemm(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_gemm, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_gemm, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}

}  // namespace pg

using namespace pg;

extern "C" pg_status pg_gemm_bf16(int64_t M, int64_t N, int64_t K, const void* A, int32_t a_mn,
                                  int64_t lda, const void* B, int32_t b_mn, int64_t ldb, void* C,
                                  pg_dtype c_dtype, int64_t ldc, int32_t accumulate,
                                  pg_stream_t stream) {
  if (M < 1 || N < 1 || K < 1 || M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31) ||
      !A || !B || !C || (a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1) ||
      (c_dtype != PG_F32 && c_dtype != PG_BF16) || (accumulate != 0 && accumulate != 1)) {
    set_error("pg_gemm_bf16: bad sizes, NULL pointer or bad layout flag");
    return PG_ERR_INVALID_ARG;
  }
  if (lda % 8 || ldb % 8 || lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N) {
    set_error("pg_gemm_bf16: leading dimensions must cover the rows and be multiples of 8");
    return PG_ERR_INVALID_ARG;
  }
  CUtensorMap ta, tb;
  pg_status st = a_mn ? make_tmap_2d_bf16(&ta, A, M, K, lda * 2, 64, 64)
                      : make_tmap_2d_bf16(&ta, A, K, M, lda * 2, 64, 128);
  if (st != PG_OK) return st;
  st = b_mn ? make_tmap_2d_bf16(&tb, B, N, K, ldb * 2, 64, 64)
            : make_tmap_2d_bf16(&tb, B, K, N, ldb * 2, 64, BN);
  if (st != PG_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int m = (int)M, n = (int)N, k = (int)K;
  if (c_dtype == PG_F32) {
    if (!a_mn && !b_mn) return launch<0, 0, float>(ta, tb, C, m, n, k, ldc, accumulate, s);
    if (!a_mn && b_mn) return launch<0, 1, float>(ta, tb, C, m, n, k, ldc, accumulate, s);
    if (a_mn && !b_mn) return launch<1, 0, float>(ta, tb, C, m, n, k, ldc, accumulate, s);
    return launch<1, 1, float>(ta, tb, C, m, n, k, ldc, accumulate, s);
  }
  if (!a_mn && !b_mn) return launch<0, 0, __nv_bfloat16>(ta, tb, C, m, n, k, ldc, accumulate, s);
  if (!a_mn && b_mn) return launch<0, 1, __nv_bfloat16>(ta, tb, C, m, n, k, ldc, accumulate, s);
  if (a_mn && !b_mn) return launch<1, 0, __nv_bfloat16>(ta, tb, C, m, n, k, ldc, accumulate, s);
  return launch<1, 1, __nv_bfloat16>(ta, tb, C, m, n, k, ldc, accumulate, s);
}

extern "C" pg_status pg_gemm_bf16_rope(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                       const void* B, int64_t ldb, void* C, int64_t ldc,
                                       int32_t head_dim, const void* table,
                                       int64_t table_rows, pg_stream_t stream) {
  if (M < 1 || N < 1 || K < 1 || M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31) ||
      !A || !B || !C || !table || table_rows < M) {
    set_error("pg_gemm_bf16_rope: bad sizes, NULL pointer or a table with fewer than M rows");
    return PG_ERR_INVALID_ARG;
  }
  if ((head_dim != 64 && head_dim != 128) || N % head_dim != 0) {
    set_error("pg_gemm_bf16_rope: head_dim must be 64 or 128 and divide N");
    return PG_ERR_INVALID_ARG;
  }
  if (lda % 8 || ldb % 8 || ldc % 8 || lda < K || ldb < K || ldc < N ||
      (reinterpret_cast<uintptr_t>(C) & 15u) || (reinterpret_cast<uintptr_t>(table) & 15u)) {
    set_error("pg_gemm_bf16_rope: leading dimensions must be multiples of 8 covering the rows, "
              "C and the table 16-byte aligned");
    return PG_ERR_INVALID_ARG;
  }
  CUtensorMap ta, tb;
  pg_status st = make_tmap_2d_bf16(&ta, A, K, M, lda * 2, 64, 128);
  if (st != PG_OK) return st;
  st = make_tmap_2d_bf16(&tb, B, K, N, ldb * 2, 64, BN);
  if (st != PG_OK) return st;
  return launch<0, 0, __nv_bfloat16, true>(ta, tb, C, (int)M, (int)N, (int)K, ldc, 0,
                                           reinterpret_cast<cudaStream_t>(stream),
                                           static_cast<const float2*>(table), head_dim);
}
