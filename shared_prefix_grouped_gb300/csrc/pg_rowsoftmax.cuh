// Row softmax pieces shared by the 128-key attention forwards (training and scoring): one thread
// owns one query row (a TMEM lane) and handles a 128-key score tile 64 columns at a time.  Scores
// arrive raw (the softmax scale, in log2 units, is folded into the exponent); P is rounded to
// bf16 and written over the scores' own TMEM columns, where the P V product reads it.
#pragma once
#include <math.h>
#include <stdint.h>

#include "pg_sm100.cuh"

namespace pg {
namespace rowsoftmax {

using namespace sm100;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 64 consecutive fp32 columns of this thread's TMEM lane into registers.
__device__ __forceinline__ void load64(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_ld_wait();
}

// Max of 64 raw scores (columns c0 .. c0 + 63 of the tile); with kMasked, columns outside the
// visible run [lo, lo + len) count as -inf.  Two columns per three-input max.
template <bool kMasked>
__device__ __forceinline__ float max64(const uint32_t (&r)[64], int c0, int lo, int len) {
  float mx = -INFINITY;
#pragma unroll
  for (int cc = 0; cc < 64; cc += 2) {
    float x0 = __uint_as_float(r[cc]), x1 = __uint_as_float(r[cc + 1]);
    if (kMasked) {
      x0 = (unsigned)(c0 + cc - lo) < (unsigned)len ? x0 : -INFINITY;
      x1 = (unsigned)(c0 + cc + 1 - lo) < (unsigned)len ? x1 : -INFINITY;
    }
    mx = fmax3(mx, x0, x1);
  }
  return mx;
}

// P = exp2(s * scale_log2 - mref) of 64 columns (c0 ..), rounded to bf16 and stored to TMEM
// columns [p_addr, p_addr + 32); returns the sum of the fp32 values (even and odd columns summed
// separately, then added).  The scale-and-shift and the sums run on column pairs.
template <bool kMasked>
__device__ __forceinline__ float exp64(const uint32_t (&r)[64], int c0, int lo, int len,
                                       float scale_log2, float mref, uint32_t p_addr) {
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-mref, -mref);
  uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pw[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const int cc = 32 * h + 2 * e;
      float x0 = __uint_as_float(r[cc]), x1 = __uint_as_float(r[cc + 1]);
      if (kMasked) {
        x0 = (unsigned)(c0 + cc - lo) < (unsigned)len ? x0 : -INFINITY;
        x1 = (unsigned)(c0 + cc + 1 - lo) < (unsigned)len ? x1 : -INFINITY;
      }
      float a0, a1;
      f2_unpack(f2_fma(f2_pack(x0, x1), sc2, nm2), a0, a1);
      const float p0 = ex2(a0);
      const float p1 = ex2(a1);
      sum2 = f2_add(sum2, f2_pack(p0, p1));
      pw[e] = pack_bf16x2(p0, p1);
    }
    tmem_st16(p_addr + 16 * h, pw);
  }
  float s0, s1;
  f2_unpack(sum2, s0, s1);
  return s0 + s1;
}

// As exp64 with the running reference, but P stays in registers (pw) and the raw max of the
// visible columns is folded into mx: the steady-state pass, whose P is stored only if no row's
// max has grown past the rescale threshold.
template <bool kMasked>
__device__ __forceinline__ float exp64_keep(const uint32_t (&r)[64], int c0, int lo, int len,
                                            float scale_log2, float mref, uint32_t (&pw)[32],
                                            float& mx) {
  const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-mref, -mref);
  uint64_t sum2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    float x0 = __uint_as_float(r[2 * e]), x1 = __uint_as_float(r[2 * e + 1]);
    if (kMasked) {
      x0 = (unsigned)(c0 + 2 * e - lo) < (unsigned)len ? x0 : -INFINITY;
      x1 = (unsigned)(c0 + 2 * e + 1 - lo) < (unsigned)len ? x1 : -INFINITY;
    }
    mx = fmax3(mx, x0, x1);
    float a0, a1;
    f2_unpack(f2_fma(f2_pack(x0, x1), sc2, nm2), a0, a1);
    const float p0 = ex2(a0);
    const float p1 = ex2(a1);
    sum2 = f2_add(sum2, f2_pack(p0, p1));
    pw[e] = pack_bf16x2(p0, p1);
  }
  float s0, s1;
  f2_unpack(sum2, s0, s1);
  return s0 + s1;
}

}  // namespace rowsoftmax
}  // namespace pg
