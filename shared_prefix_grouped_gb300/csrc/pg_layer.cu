// Element-wise and row-wise kernels of the decoder layer: RMSNorm (with the residual add fused in
// front of it) forward and backward, and SwiGLU forward and backward.  Activations are bf16,
// arithmetic fp32; the RMSNorm weight gradient is reduced deterministically (fixed-order partial
// sums per block of rows, then a fixed-order sum of the partials).
#include <math.h>

#include <algorithm>

#include "pg_internal.h"

namespace pg {

namespace {

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float block_sum(float v, float* red) {
  // blockDim.x == 256
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += red[i];
  return s;
}

// y = x (+ res); out = y * rstd * gamma with rstd = 1 / sqrt(mean(y^2) + eps); sum_out = y.
// One block of 256 threads per row.
__global__ void __launch_bounds__(256)
rmsnorm_fwd_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ res,
                   const __nv_bfloat16* __restrict__ gamma, float eps, int hidden,
                   __nv_bfloat16* __restrict__ out, __nv_bfloat16* __restrict__ sum_out,
                   float* __restrict__ rstd_out) {
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const __nv_bfloat16* xr = x + row * hidden;
  float ss = 0.f;
  for (int c = threadIdx.x; c < hidden; c += 256) {
    float y = bf(xr[c]);
    if (res) {
      // the residual sum is stored in bf16 and normalised as stored
      y = bf(__float2bfloat16_rn(y + bf(res[row * hidden + c])));
      sum_out[row * hidden + c] = __float2bfloat16_rn(y);
    }
    ss += y * y;
  }
  const float rstd = rsqrtf(block_sum(ss, red) / hidden + eps);
  for (int c = threadIdx.x; c < hidden; c += 256) {
    const float y = res ? bf(sum_out[row * hidden + c]) : bf(xr[c]);
    out[row * hidden + c] = __float2bfloat16_rn(y * rstd * bf(gamma[c]));
  }
  if (threadIdx.x == 0) rstd_out[row] = rstd;
}

// dx = dres + rstd * (gamma*dout - yhat * mean(yhat * gamma*dout)), yhat = y * rstd, for a block
// of ROWS rows; the block's partial sum of dout * yhat (the gamma gradient) goes to
// dgamma_part[blockIdx.x][hidden].  dout is fp32 or bf16; dres (optional) bf16; dx bf16 or fp32.
constexpr int RN_ROWS = 16;

template <typename DoutT, typename DxT>
__global__ void __launch_bounds__(256)
rmsnorm_bwd_kernel(const __nv_bfloat16* __restrict__ y, const __nv_bfloat16* __restrict__ gamma,
                   const float* __restrict__ rstd, const DoutT* __restrict__ dout,
                   const __nv_bfloat16* __restrict__ dres, DxT* __restrict__ dx,
                   float* __restrict__ dgamma_part, int T, int hidden) {
  extern __shared__ float dg[];   // [hidden]
  __shared__ float red[8];
  for (int c = threadIdx.x; c < hidden; c += 256) dg[c] = 0.f;
  const int r0 = blockIdx.x * RN_ROWS;
  for (int row = r0; row < min(r0 + RN_ROWS, T); ++row) {
    const size_t base = (size_t)row * hidden;
    const float rs = rstd[row];
    float dot = 0.f;
    for (int c = threadIdx.x; c < hidden; c += 256) {
      const float yh = bf(y[base + c]) * rs;
      const float gd = bf(gamma[c]) * (float)dout[base + c];
      dot += yh * gd;
    }
    const float mean = block_sum(dot, red) / hidden;
    for (int c = threadIdx.x; c < hidden; c += 256) {
      const float yh = bf(y[base + c]) * rs;
      const float d = (float)dout[base + c];
      float g = rs * (bf(gamma[c]) * d - yh * mean);
      if (dres) g += bf(dres[base + c]);
      if constexpr (sizeof(DxT) == 4) dx[base + c] = g;
      else dx[base + c] = __float2bfloat16_rn(g);
      dg[c] += d * yh;
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < hidden; c += 256)
    dgamma_part[(size_t)blockIdx.x * hidden + c] = dg[c];
}

__global__ void sum_partials_kernel(const float* __restrict__ part, int nparts, int hidden,
                                    float* __restrict__ out) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= hidden) return;
  float s = 0.f;
  for (int p = 0; p < nparts; ++p) s += part[(size_t)p * hidden + c];
  out[c] = s;
}

__device__ __forceinline__ float sigmoidf_(float g) { return 1.f / (1.f + expf(-g)); }

// gu = [gate | up] rows of width 2I; out = silu(gate) * up.
__global__ void swiglu_fwd_kernel(const __nv_bfloat16* __restrict__ gu, int I, size_t n,
                                  __nv_bfloat16* __restrict__ out) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t t = e / I, i = e - t * I;
    const float g = bf(gu[t * 2 * I + i]), u = bf(gu[t * 2 * I + I + i]);
    out[e] = __float2bfloat16_rn(g * sigmoidf_(g) * u);
  }
}

// d_gate = d_out * up * sigma(g) * (1 + g * (1 - sigma(g))), d_up = d_out * silu(g).
__global__ void swiglu_bwd_kernel(const __nv_bfloat16* __restrict__ gu,
                                  const __nv_bfloat16* __restrict__ dout, int I, size_t n,
                                  __nv_bfloat16* __restrict__ dgu) {
  for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (size_t)gridDim.x * blockDim.x) {
    const size_t t = e / I, i = e - t * I;
    const float g = bf(gu[t * 2 * I + i]), u = bf(gu[t * 2 * I + I + i]);
    const float d = bf(dout[e]);
    const float sg = sigmoidf_(g);
    dgu[t * 2 * I + i] = __float2bfloat16_rn(d * u * sg * (1.f + g * (1.f - sg)));
    dgu[t * 2 * I + I + i] = __float2bfloat16_rn(d * g * sg);
  }
}

}  // namespace

}  // namespace pg

using namespace pg;

extern "C" {

pg_status pg_rmsnorm_fwd(int64_t T, int32_t hidden, const void* x, const void* residual,
                         const void* gamma, float eps, void* out, void* sum_out, float* rstd,
                         pg_stream_t stream) {
  if (T < 1 || hidden < 1 || hidden > (1 << 16) || !x || !gamma || !out || !rstd || eps < 0.f ||
      (residual && !sum_out)) {
    set_error("pg_rmsnorm_fwd: bad sizes or pointers (sum_out is required with a residual)");
    return PG_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  prof_begin(PG_KERNEL_LAYER, s);
  rmsnorm_fwd_kernel<<<(unsigned)T, 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(residual),
      static_cast<const __nv_bfloat16*>(gamma), eps, hidden, static_cast<__nv_bfloat16*>(out),
      static_cast<__nv_bfloat16*>(sum_out), rstd);
  prof_end(PG_KERNEL_LAYER, s);
  return cuda_check(cudaGetLastError(), "rmsnorm fwd launch");
}

size_t pg_rmsnorm_bwd_workspace(int64_t T, int32_t hidden) {
  const int64_t nb = (T + RN_ROWS - 1) / RN_ROWS;
  return (size_t)nb * hidden * sizeof(float);
}

pg_status pg_rmsnorm_bwd(int64_t T, int32_t hidden, const void* y, const void* gamma,
                         const float* rstd, const void* dout, pg_dtype dout_dtype,
                         const void* dres, void* dx, pg_dtype dx_dtype, float* dgamma,
                         void* workspace, size_t workspace_bytes, pg_stream_t stream) {
  if (T < 1 || hidden < 1 || hidden > 12288 || !y || !gamma || !rstd || !dout || !dx || !dgamma ||
      !workspace || workspace_bytes < pg_rmsnorm_bwd_workspace(T, hidden) ||
      (dout_dtype != PG_F32 && dout_dtype != PG_BF16) || (dx_dtype != PG_F32 && dx_dtype != PG_BF16)) {
    set_error("pg_rmsnorm_bwd: bad sizes, pointers, dtypes or workspace");
    return PG_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t nb = (T + RN_ROWS - 1) / RN_ROWS;
  float* part = static_cast<float*>(workspace);
  const size_t smem = (size_t)hidden * sizeof(float);
  const auto* yy = static_cast<const __nv_bfloat16*>(y);
  const auto* gg = static_cast<const __nv_bfloat16*>(gamma);
  const auto* rr = static_cast<const __nv_bfloat16*>(dres);
  prof_begin(PG_KERNEL_LAYER, s);
#define PG_RN_LAUNCH(DO, DX)                                                                    \
  do {                                                                                          \
    auto k = rmsnorm_bwd_kernel<DO, DX>;                                                        \
    pg_status st_ = cuda_check(                                                                 \
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),       \
        "rmsnorm bwd smem");                                                                    \
    if (st_ != PG_OK) return st_;                                                               \
    k<<<(unsigned)nb, 256, smem, s>>>(yy, gg, rstd, static_cast<const DO*>(dout), rr,           \
                                     static_cast<DX*>(dx), part, (int)T, hidden);               \
  } while (0)
  if (dout_dtype == PG_F32 && dx_dtype == PG_F32) PG_RN_LAUNCH(float, float);
  else if (dout_dtype == PG_F32) PG_RN_LAUNCH(float, __nv_bfloat16);
  else if (dx_dtype == PG_F32) PG_RN_LAUNCH(__nv_bfloat16, float);
  else PG_RN_LAUNCH(__nv_bfloat16, __nv_bfloat16);
#undef PG_RN_LAUNCH
  sum_partials_kernel<<<(hidden + 255) / 256, 256, 0, s>>>(part, (int)nb, hidden, dgamma);
  prof_end(PG_KERNEL_LAYER, s);
  return cuda_check(cudaGetLastError(), "rmsnorm bwd launch");
}

pg_status pg_swiglu_fwd(int64_t T, int32_t inter, const void* gate_up, void* out,
                        pg_stream_t stream) {
  if (T < 1 || inter < 1 || !gate_up || !out) {
    set_error("pg_swiglu_fwd: bad sizes or pointers");
    return PG_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t n = (size_t)T * inter;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 152 * 32);
  prof_begin(PG_KERNEL_LAYER, s);
  swiglu_fwd_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(gate_up), inter, n,
                                           static_cast<__nv_bfloat16*>(out));
  prof_end(PG_KERNEL_LAYER, s);
  return cuda_check(cudaGetLastError(), "swiglu fwd launch");
}

pg_status pg_swiglu_bwd(int64_t T, int32_t inter, const void* gate_up, const void* dout,
                        void* dgate_up, pg_stream_t stream) {
  if (T < 1 || inter < 1 || !gate_up || !dout || !dgate_up) {
    set_error("pg_swiglu_bwd: bad sizes or pointers");
    return PG_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t n = (size_t)T * inter;
  const unsigned blocks = (unsigned)std::min<size_t>((n + 255) / 256, 152 * 32);
  prof_begin(PG_KERNEL_LAYER, s);
  swiglu_bwd_kernel<<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(gate_up),
                                           static_cast<const __nv_bfloat16*>(dout), inter, n,
                                           static_cast<__nv_bfloat16*>(dgate_up));
  prof_end(PG_KERNEL_LAYER, s);
  return cuda_check(cudaGetLastError(), "swiglu bwd launch");
}

}  // extern "C"
