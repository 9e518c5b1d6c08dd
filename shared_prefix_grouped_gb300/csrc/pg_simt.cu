// SIMT kernels of the grouped-attention library: RoPE, the fp32-arithmetic attention forward and
// backward (exact fp32 FFMA, no tensor cores), and the backward preprocess.
//
// The attention kernels evaluate, for every packed query row t, softmax attention over the keys s
// with  s <= t && s >= g0 && (s < pe || s >= own_lo(t))  -- the prefix causally for prefix rows,
// the whole prefix plus the row's own response for response rows (Pith review of Prefix Grouper,
// "What carries the argument").  Work is organised per tile of 64 rows of one group; each tile
// visits two key ranges: the group's prefix, then the responses' part that its rows can see.
//
// Thread layout: 4 threads ("a quad") per row; quad lane ql holds head-dim elements
// {4*ql + 16*i + c : i < d/16, c < 4}, so a row's dot product is a 4-lane shuffle reduction and a
// shared-memory row read by a warp touches 64 consecutive bytes (no bank conflicts).  Dimension k
// and k + d/2 live in the same lane (d/2 is a multiple of 16).
#include <math.h>

#include <algorithm>

#include "pg_internal.h"

namespace pg {

namespace {

__device__ int s_status_simt = 0;

__device__ __forceinline__ void report(int code) { atomicCAS(&s_status_simt, 0, code); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T>
struct Vec;

template <>
struct Vec<float> {
  static __device__ __forceinline__ float4 load4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
  }
  static __device__ __forceinline__ void store4(float* p, float4 v) {
    *reinterpret_cast<float4*>(p) = v;
  }
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store(float* p, float v) { *p = v; }
  static __device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
  static __device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
};

template <>
struct Vec<__nv_bfloat16> {
  static __device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    uint2 u = *reinterpret_cast<const uint2*>(p);
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&u.x);
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&u.y);
    float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
  }
  static __device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
  }
  static __device__ __forceinline__ float load(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
  static __device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  return x;
}

// ---------------------------------------------------------------------------------------------
// RoPE: rotate (or inverse-rotate) the pairs (x[k], x[k + d/2]) of every head of a token by the
// angle pos * theta^(-2k/d).  The inverse frequencies come from the host in fp64; the angle is
// formed and reduced to [-pi, pi] in fp64 (two multiplies and a rounding), then sin/cos are taken
// in fp32.  With a table_out the (cos, sin) pairs are also stored ([T][d/2] float2) for later
// passes of the same call; with a table_in they are read from it instead of recomputed.
// `rope` false only converts (used to cast the fp32 gradient accumulators).
// A block handles `tpb` consecutive tokens (enough to give its 256 threads 16-byte chunks of work
// when a token has few heads); two tensors (q and k) per launch.  With `spans` (the layout's
// response spans) the blocks cover only the response tokens: `span_blocks` blocks per span.
// ---------------------------------------------------------------------------------------------
constexpr int kRopeThreads = 256;
constexpr int kRopeMaxTokens = 8;

// 2 pi / 2^32: one unit of a turn's upper 32 fraction bits, in radians.
constexpr float kRadPerTurnUnit = 1.4629180792671596e-09f;

// With bf16 input a thread needs at most 32 registers, so eight blocks fit on an SM: the pass is
// bound by the bytes each SM keeps in flight.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kRopeThreads, sizeof(Tin) == 2 ? 8 : 6)
rope_kernel(const Tin* __restrict__ x0, Tout* __restrict__ y0, int h0,
            const Tin* __restrict__ x1, Tout* __restrict__ y1, int h1, int d, int Ttot, int tpb,
            const FwdTile* __restrict__ spans, int span_blocks, int split, int tpb1,
            const int32_t* __restrict__ pos_ids, RopeFreq f, int rope, float sgn,
            float2* __restrict__ table_out, const float2* __restrict__ table_in) {
  __shared__ float cs[kRopeMaxTokens][64], sn[kRopeMaxTokens][64];
  int blk = blockIdx.x;
  if (split > 0) {
    // Two parts: blocks [0, split) rotate every row of x0, the others the response rows of x1.
    if (blk >= split) {
      blk -= split;
      x0 = x1;
      y0 = y1;
      h0 = h1;
      tpb = tpb1;
    } else {
      spans = nullptr;
    }
    h1 = 0;
  }
  int t_first = blk * tpb, t_limit = Ttot;
  if (spans != nullptr) {
    const FwdTile sp = spans[blk / span_blocks];
    t_first = sp.q0 + (blk % span_blocks) * tpb;
    t_limit = min(sp.q1, Ttot);
    if (t_first >= t_limit) return;
  }
  const int half = d >> 1;
  for (int e = threadIdx.x; e < tpb * half; e += blockDim.x) {
    const int tl = e / half, k = e - tl * half, t = t_first + tl;
    float c = 1.f, s = 0.f;
    if (rope && t < t_limit) {
      if (table_in) {
        const float2 v = table_in[(size_t)t * half + k];
        c = v.x;
        s = v.y;
      } else {
        // position x (inv_freq / 2 pi) modulo one turn, exact in 0.64 fixed point (positions
        // are non-negative); its upper 32 bits read as signed give the angle in [-pi, pi).
        const uint64_t turns = (uint64_t)(uint32_t)pos_ids[t] * f.turn[k];
        const float r = (float)(int32_t)(uint32_t)(turns >> 32) * kRadPerTurnUnit;
        sincosf(r, &s, &c);
        if (table_out) table_out[(size_t)t * half + k] = make_float2(c, s);
      }
    }
    cs[tl][k] = c;
    sn[tl][k] = sgn * s;
  }
  __syncthreads();
  // Each work item rotates 8 consecutive pairs of one head of one token (16-byte loads of bf16,
  // 32-byte of fp32).
  const int chunks = half >> 3;
  for (int which = 0; which < 2; ++which) {
    const Tin* x = which ? x1 : x0;
    Tout* y = which ? y1 : y0;
    const int heads = which ? h1 : h0;
    const int per_token = heads * chunks;
    for (int idx = threadIdx.x; idx < tpb * per_token; idx += blockDim.x) {
      const int tl = idx / per_token, rem = idx - tl * per_token, t = t_first + tl;
      if (t >= t_limit) break;
      const int h = rem / chunks, k0 = (rem - h * chunks) * 8;
      const size_t i1 = ((size_t)t * heads + h) * d + k0;
      float a[8], b[8], lo[8], hi[8];
      Vec<Tin>::load8(x + i1, a);
      Vec<Tin>::load8(x + i1 + half, b);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float c = cs[tl][k0 + e], s = sn[tl][k0 + e];
        lo[e] = a[e] * c - b[e] * s;
        hi[e] = b[e] * c + a[e] * s;
      }
      Vec<Tout>::store8(y + i1, lo);
      Vec<Tout>::store8(y + i1 + half, hi);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// Forward: online softmax over the tile's key ranges, 64 keys at a time staged in shared memory.
// ---------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, const int4* __restrict__ tok,
                const FwdTile* __restrict__ tiles, const int2* __restrict__ ivs, int Hq, int Hkv,
                int Ttot, float qscale, int responses_only) {
  constexpr int BN = 64, NV = D / 16;
  extern __shared__ float4 smem4[];
  float* Ks = reinterpret_cast<float*>(smem4);
  float* Vs = Ks + BN * D;
  const int tile_id = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const FwdTile tl = tiles[tile_id];
  if (tl.q0 < 0 || tl.q1 > Ttot || tl.q0 >= tl.q1 || tl.g0 < 0 || tl.s_hi > Ttot ||
      tl.a_cnt < 0 || tl.a_cnt > kMaxExtraRanges) {
    report(PG_ERR_DEVICE);
    return;
  }
  // Responses only (two-level layouts): a row before its group's prefix end (the token table's
  // pe) is a prefix row and computes nothing; a tile of prefix rows exits at once (uniformly).
  if (responses_only && tl.q1 <= tok[tl.q1 - 1].y) return;
  const int kh = h / (Hq / Hkv);
  const int tid = threadIdx.x, r = tid >> 2, ql = tid & 3;
  const int row = tl.q0 + r;
  const int4 tr_ = tok[row < tl.q1 ? row : tl.q1 - 1];
  const bool valid = row < tl.q1 && !(responses_only && row < tr_.y);
  const int rowc = valid ? row : tl.q1 - 1;
  const int4 ti = tok[rowc];
  KeyRanges kr;
  kr.init(tl, ivs);
  float4 qv[NV], acc[NV];
  const T* qrow = q + ((size_t)rowc * Hq + h) * D + 4 * ql;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float4 x = Vec<T>::load4(qrow + 16 * i);
    qv[i] = make_float4(x.x * qscale, x.y * qscale, x.z * qscale, x.w * qscale);
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;
  for (int range = 0; range < kr.n; ++range) {
    const int lo = kr.lo[range], hi = kr.hi[range];
    const bool own = range >= kr.n_causal;   // own range: keys from the row's own segment only
    for (int kt = lo; kt < hi; kt += BN) {
      __syncthreads();
      for (int e = tid; e < BN * D / 4; e += 256) {
        int j = e / (D / 4), c = (e % (D / 4)) * 4;
        int key = kt + j;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
        if (key < hi) {
          size_t off = ((size_t)key * Hkv + kh) * D + c;
          kk = Vec<T>::load4(k + off);
          vv = Vec<T>::load4(v + off);
        }
        *reinterpret_cast<float4*>(Ks + j * D + c) = kk;
        *reinterpret_cast<float4*>(Vs + j * D + c) = vv;
      }
      __syncthreads();
      float s[BN];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        float p = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i)
          p += dot4(qv[i], *reinterpret_cast<const float4*>(Ks + j * D + 4 * ql + 16 * i));
        p = quad_sum(p);
        int key = kt + j;
        s[j] = (key < hi && key <= rowc && (!own || key >= ti.z)) ? p : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
      const float mnew = fmaxf(m, mt);
      const float mref = (mnew == -INFINITY) ? 0.f : mnew;
      const float corr = exp2f(m - mref);
      l *= corr;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        acc[i].x *= corr; acc[i].y *= corr; acc[i].z *= corr; acc[i].w *= corr;
      }
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        const float p = exp2f(s[j] - mref);
        l += p;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          float4 vv = *reinterpret_cast<const float4*>(Vs + j * D + 4 * ql + 16 * i);
          acc[i].x = fmaf(p, vv.x, acc[i].x);
          acc[i].y = fmaf(p, vv.y, acc[i].y);
          acc[i].z = fmaf(p, vv.z, acc[i].z);
          acc[i].w = fmaf(p, vv.w, acc[i].w);
        }
      }
      m = mnew;
    }
  }
  if (valid) {
    const float inv = 1.f / l;
    T* orow = o + ((size_t)row * Hq + h) * D + 4 * ql;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      Vec<T>::store4(orow + 16 * i,
                     make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv));
    if (ql == 0) lse[(size_t)h * Ttot + row] = (m + log2f(l)) * kLn2;
  }
}

// ---------------------------------------------------------------------------------------------
// Backward preprocess: Dbuf[h][t] = sum_j dO[t,h,j] * O[t,h,j] and lse2[h][t] = lse[h][t] * log2 e
// (fp32 rows of stride ldd >= T, padding zeroed), and zero the fp32 dQ accumulator.
// One warp per (t, h).
// ---------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
bwd_pre_kernel(const T* __restrict__ o, const T* __restrict__ dO, const float* __restrict__ lse,
               float* __restrict__ Dbuf, float* __restrict__ lse2, float* __restrict__ dq_acc,
               int Hq, int D, int Ttot, int ldd, int lse2_ready) {
  // D / 8 lanes per (t, h) row, 8 elements each (16-byte loads of bf16), so a warp covers 2 or 4
  // rows with every load in flight at once.
  const int lpr = D >> 3;                        // lanes per row
  const int lane = threadIdx.x & 31;
  const size_t gthread = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t row = gthread / lpr;              // over ldd * Hq rows, t-major
  const int sub = (int)(gthread % lpr);
  const bool in = row < (size_t)ldd * Hq;
  const int t = in ? (int)(row / Hq) : 0, h = in ? (int)(row % Hq) : 0;
  float acc = 0.f;
  if (in && t < Ttot) {
    const size_t base = ((size_t)t * Hq + h) * D + 8 * sub;
    float a[8], b[8];
    Vec<T>::load8(o + base, a);
    Vec<T>::load8(dO + base, b);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(a[e], b[e], acc);
    if (dq_acc) {
      float4* z = reinterpret_cast<float4*>(dq_acc + base);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in && sub == 0) {
    const size_t idx = (size_t)h * ldd + t;
    if (t >= Ttot) {                             // padding rows of the fp32 row buffers
      Dbuf[idx] = 0.f;
      lse2[idx] = 0.f;
    } else {
      Dbuf[idx] = acc;
      if (!lse2_ready) lse2[idx] = lse[(size_t)h * Ttot + t] * kLog2e;
    }
  }
  (void)lane;
}

// ---------------------------------------------------------------------------------------------
// dK / dV, key-major: a block owns 64 keys of one KV head and sweeps, in a fixed order, every
// query head of the KV head and every query row that can see its keys.  For a prefix key that is
// the rest of the prefix and then all responses of the group, so the cross-response sum of the
// prefix gradient happens inside one block in a fixed order (deterministic, no atomics).
// ---------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256)
dkdv_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                 const T* __restrict__ dO, const float* __restrict__ lse,
                 const float* __restrict__ Dbuf, float* __restrict__ dk_acc, T* __restrict__ dv,
                 const int4* __restrict__ tok, const BwdTile* __restrict__ tiles, int Hq, int Hkv,
                 int Ttot, int ldd, float scale_log2, float scale) {
  constexpr int BM = 64, NV = D / 16;
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);
  float* dOs = Qs + BM * D;
  float* Ls = dOs + BM * D;
  float* Ds = Ls + BM;
  int4* Ts = reinterpret_cast<int4*>(Ds + BM);
  const int tile_id = blockIdx.x / Hkv, kh = blockIdx.x % Hkv;
  const BwdTile tl = tiles[tile_id];
  if (tl.k0 < 0 || tl.k1 > Ttot || tl.k0 >= tl.k1 || tl.q_lo < 0 || tl.q_hi > Ttot) {
    report(PG_ERR_DEVICE);
    return;
  }
  const int tid = threadIdx.x, r = tid >> 2, ql = tid & 3;
  const int key = tl.k0 + r;
  const bool valid = key < tl.k1;
  const int keyc = valid ? key : tl.k1 - 1;
  float4 kv[NV], vv[NV], dk[NV], dvv[NV];
  const size_t kvoff = ((size_t)keyc * Hkv + kh) * D + 4 * ql;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float4 a = Vec<T>::load4(k + kvoff + 16 * i);
    kv[i] = make_float4(a.x * scale_log2, a.y * scale_log2, a.z * scale_log2, a.w * scale_log2);
    vv[i] = Vec<T>::load4(v + kvoff + 16 * i);
    dk[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    dvv[i] = dk[i];
  }
  const int rep = Hq / Hkv;
  for (int hh = 0; hh < rep; ++hh) {
    const int h = kh * rep + hh;
    for (int qt = tl.q_lo; qt < tl.q_hi; qt += BM) {
      __syncthreads();
      for (int e = tid; e < BM * D / 4; e += 256) {
        int j = e / (D / 4), c = (e % (D / 4)) * 4;
        int qr = qt + j;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (qr < tl.q_hi) {
          size_t off = ((size_t)qr * Hq + h) * D + c;
          a = Vec<T>::load4(q + off);
          b = Vec<T>::load4(dO + off);
        }
        *reinterpret_cast<float4*>(Qs + j * D + c) = a;
        *reinterpret_cast<float4*>(dOs + j * D + c) = b;
      }
      if (tid < BM) {
        int qr = qt + tid;
        bool in = qr < tl.q_hi;
        Ls[tid] = in ? lse[(size_t)h * Ttot + qr] * kLog2e : 0.f;
        Ds[tid] = in ? Dbuf[(size_t)h * ldd + qr] : 0.f;
        Ts[tid] = in ? tok[qr] : make_int4(0, 0, 0, 0);
      }
      __syncthreads();
      const int jn = min(BM, tl.q_hi - qt);
      for (int j = 0; j < jn; ++j) {
        const int qr = qt + j;
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          s += dot4(kv[i], *reinterpret_cast<const float4*>(Qs + j * D + 4 * ql + 16 * i));
          dp += dot4(vv[i], *reinterpret_cast<const float4*>(dOs + j * D + 4 * ql + 16 * i));
        }
        s = quad_sum(s);
        dp = quad_sum(dp);
        // Key-major visibility of a tile: rows [keyc, q_hi) see the key if it is a prefix-like
        // key of the tile (keyc < pe) or lies in the row's own segment.
        const bool vis = valid && keyc <= qr && qr < tl.q_hi && (keyc < tl.pe || keyc >= Ts[j].z);
        const float p = vis ? exp2f(s - Ls[j]) : 0.f;
        const float ds = p * (dp - Ds[j]);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          float4 a = *reinterpret_cast<const float4*>(Qs + j * D + 4 * ql + 16 * i);
          float4 b = *reinterpret_cast<const float4*>(dOs + j * D + 4 * ql + 16 * i);
          dvv[i].x = fmaf(p, b.x, dvv[i].x); dvv[i].y = fmaf(p, b.y, dvv[i].y);
          dvv[i].z = fmaf(p, b.z, dvv[i].z); dvv[i].w = fmaf(p, b.w, dvv[i].w);
          dk[i].x = fmaf(ds, a.x, dk[i].x); dk[i].y = fmaf(ds, a.y, dk[i].y);
          dk[i].z = fmaf(ds, a.z, dk[i].z); dk[i].w = fmaf(ds, a.w, dk[i].w);
        }
      }
    }
  }
  if (valid) {
    const size_t off = ((size_t)key * Hkv + kh) * D + 4 * ql;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      *reinterpret_cast<float4*>(dk_acc + off + 16 * i) =
          make_float4(dk[i].x * scale, dk[i].y * scale, dk[i].z * scale, dk[i].w * scale);
      Vec<T>::store4(dv + off + 16 * i, dvv[i]);
    }
  }
}

// ---------------------------------------------------------------------------------------------
// dQ, query-major: recomputes P and dP for the tile's rows over the same key ranges as the
// forward and writes scale * sum_s dS[t,s] k_s (fp32, rotated frame).
// ---------------------------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256)
dq_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
               const T* __restrict__ dO, const float* __restrict__ lse,
               const float* __restrict__ Dbuf, float* __restrict__ dq_acc,
               const int4* __restrict__ tok, const FwdTile* __restrict__ tiles,
               const int2* __restrict__ ivs, int Hq, int Hkv, int Ttot, int ldd, float scale_log2,
               float scale) {
  constexpr int BN = 64, NV = D / 16;
  extern __shared__ float4 smem4[];
  float* Ks = reinterpret_cast<float*>(smem4);
  float* Vs = Ks + BN * D;
  const int tile_id = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const FwdTile tl = tiles[tile_id];
  if (tl.q0 < 0 || tl.q1 > Ttot || tl.q0 >= tl.q1 || tl.g0 < 0 || tl.s_hi > Ttot ||
      tl.a_cnt < 0 || tl.a_cnt > kMaxExtraRanges) {
    report(PG_ERR_DEVICE);
    return;
  }
  KeyRanges kr;
  kr.init(tl, ivs);
  const int kh = h / (Hq / Hkv);
  const int tid = threadIdx.x, r = tid >> 2, ql = tid & 3;
  const int row = tl.q0 + r;
  const bool valid = row < tl.q1;
  const int rowc = valid ? row : tl.q1 - 1;
  const int4 ti = tok[rowc];
  float4 qv[NV], dov[NV], dq[NV];
  const size_t qoff = ((size_t)rowc * Hq + h) * D + 4 * ql;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    float4 a = Vec<T>::load4(q + qoff + 16 * i);
    qv[i] = make_float4(a.x * scale_log2, a.y * scale_log2, a.z * scale_log2, a.w * scale_log2);
    dov[i] = Vec<T>::load4(dO + qoff + 16 * i);
    dq[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float L2 = lse[(size_t)h * Ttot + rowc] * kLog2e;
  const float Dr = Dbuf[(size_t)h * ldd + rowc];
  for (int range = 0; range < kr.n; ++range) {
    const int lo = kr.lo[range], hi = kr.hi[range];
    const bool own = range >= kr.n_causal;
    for (int kt = lo; kt < hi; kt += BN) {
      __syncthreads();
      for (int e = tid; e < BN * D / 4; e += 256) {
        int j = e / (D / 4), c = (e % (D / 4)) * 4;
        int key = kt + j;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), vv = kk;
        if (key < hi) {
          size_t off = ((size_t)key * Hkv + kh) * D + c;
          kk = Vec<T>::load4(k + off);
          vv = Vec<T>::load4(v + off);
        }
        *reinterpret_cast<float4*>(Ks + j * D + c) = kk;
        *reinterpret_cast<float4*>(Vs + j * D + c) = vv;
      }
      __syncthreads();
      const int jn = min(BN, hi - kt);
      for (int j = 0; j < jn; ++j) {
        float s = 0.f, dp = 0.f;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          s += dot4(qv[i], *reinterpret_cast<const float4*>(Ks + j * D + 4 * ql + 16 * i));
          dp += dot4(dov[i], *reinterpret_cast<const float4*>(Vs + j * D + 4 * ql + 16 * i));
        }
        s = quad_sum(s);
        dp = quad_sum(dp);
        const bool vis = kt + j <= rowc && (!own || kt + j >= ti.z);
        const float p = vis ? exp2f(s - L2) : 0.f;
        const float ds = p * (dp - Dr);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          float4 kk = *reinterpret_cast<const float4*>(Ks + j * D + 4 * ql + 16 * i);
          dq[i].x = fmaf(ds, kk.x, dq[i].x); dq[i].y = fmaf(ds, kk.y, dq[i].y);
          dq[i].z = fmaf(ds, kk.z, dq[i].z); dq[i].w = fmaf(ds, kk.w, dq[i].w);
        }
      }
    }
  }
  if (valid) {
    const size_t off = ((size_t)row * Hq + h) * D + 4 * ql;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      *reinterpret_cast<float4*>(dq_acc + off + 16 * i) =
          make_float4(dq[i].x * scale, dq[i].y * scale, dq[i].z * scale, dq[i].w * scale);
  }
}

template <typename KernelT>
pg_status set_smem(KernelT kernel, size_t bytes) {
  return cuda_check(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)bytes),
                    "cudaFuncSetAttribute(max dynamic smem)");
}

template <typename T, int D>
pg_status fwd_simt_t(const AttnArgs& a, const void* q, const void* k, const void* v, void* o,
                     float* lse) {
  const pg_layout* L = a.layout;
  const int64_t n = L->n_tiles[FWD64];
  const size_t smem = 2 * 64 * D * sizeof(float);
  auto kern = fwd_simt_kernel<T, D>;
  pg_status st = set_smem(kern, smem);
  if (st != PG_OK) return st;
  prof_begin(PG_KERNEL_ATTN_FWD, a.stream);
  kern<<<(unsigned)(n * a.Hq), 256, smem, a.stream>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
      static_cast<T*>(o), lse, tokens(L), tiles<FwdTile>(L, FWD64), intervals(L), a.Hq, a.Hkv,
      (int)L->total_tokens, a.scale * kLog2e, (a.flags & PG_FLAG_RESPONSES_ONLY) ? 1 : 0);
  prof_end(PG_KERNEL_ATTN_FWD, a.stream);
  return cuda_check(cudaGetLastError(), "fwd_simt launch");
}

template <typename T, int D>
pg_status bwd_simt_t(const AttnArgs& a, const void* q, const void* k, const void* v,
                     const void* dO, const float* lse, const float* Dbuf, float* dq_acc,
                     float* dk_acc, void* dv) {
  const pg_layout* L = a.layout;
  const int Ttot = (int)L->total_tokens;
  {
    const size_t smem = 2 * 64 * D * sizeof(float) + 64 * (2 * sizeof(float) + sizeof(int4));
    auto kern = dkdv_simt_kernel<T, D>;
    pg_status st = set_smem(kern, smem);
    if (st != PG_OK) return st;
    prof_begin(PG_KERNEL_BWD_DKDV, a.stream);
    kern<<<(unsigned)(L->n_tiles[BWD64] * a.Hkv), 256, smem, a.stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(dO), lse, Dbuf, dk_acc, static_cast<T*>(dv), tokens(L),
        tiles<BwdTile>(L, BWD64), a.Hq, a.Hkv, Ttot, (int)padded_tokens(L), a.scale * kLog2e,
        a.scale);
    prof_end(PG_KERNEL_BWD_DKDV, a.stream);
    st = cuda_check(cudaGetLastError(), "dkdv_simt launch");
    if (st != PG_OK) return st;
  }
  {
    const size_t smem = 2 * 64 * D * sizeof(float);
    auto kern = dq_simt_kernel<T, D>;
    pg_status st = set_smem(kern, smem);
    if (st != PG_OK) return st;
    prof_begin(PG_KERNEL_BWD_DQ, a.stream);
    kern<<<(unsigned)(L->n_tiles[FWD64] * a.Hq), 256, smem, a.stream>>>(
        static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v),
        static_cast<const T*>(dO), lse, Dbuf, dq_acc, tokens(L), tiles<FwdTile>(L, FWD64),
        intervals(L), a.Hq,
        a.Hkv, Ttot, (int)padded_tokens(L), a.scale * kLog2e, a.scale);
    prof_end(PG_KERNEL_BWD_DQ, a.stream);
    return cuda_check(cudaGetLastError(), "dq_simt launch");
  }
}

}  // namespace

RopeFreq rope_freq(const AttnArgs& a) {
  RopeFreq f{};
  if (a.theta > 0.f)
    for (int k = 0; k < a.d / 2 && k < 64; ++k) {
      double c = pow((double)a.theta, -2.0 * k / a.d) / 6.283185307179586476925;
      c -= floor(c);                                  // whole turns drop out of position x c
      f.turn[k] = (uint64_t)ldexp(c, 64);             // c < 1, so this is below 2^64
    }
  return f;
}

pg_status launch_rope(const AttnArgs& a, const void* x0, void* y0, int heads0, const void* x1,
                      void* y1, int heads1, bool inverse, bool in_fp32, float2* table_out,
                      const float2* table_in, RopeRows rows) {
  const int T = (int)a.layout->total_tokens;
  const int rope = a.theta > 0.f ? 1 : 0;
  const RopeFreq f = rope_freq(a);
  const float sgn = inverse ? -1.f : 1.f;
  const int32_t* pos = a.layout->position_ids;
  // Tokens per block: enough 16-byte work items (heads x d/16 per token) for the block's threads.
  auto per_block = [&](int heads) {
    const int items = heads * (a.d / 16);
    return std::max(1, std::min(kRopeMaxTokens, kRopeThreads / std::max(items, 1)));
  };
  const bool split = rows == RopeRows::kAllThenResponses;
  if (split && (x1 == nullptr || table_out != nullptr || table_in != nullptr)) {
    set_error("rope: the two-part pass takes two tensors and no cos/sin table");
    return PG_ERR_INVALID_ARG;
  }
  const int tpb = per_block(heads0 + (x1 && !split ? heads1 : 0));
  const int tpb1 = split ? per_block(heads1) : tpb;
  const FwdTile* spans = split ? tiles<FwdTile>(a.layout, SPANS) : nullptr;
  const int span_blocks =
      split ? (int)std::max<int64_t>(1, (a.layout->max_response_rows + tpb1 - 1) / tpb1) : 1;
  const int64_t all_blocks = (T + tpb - 1) / tpb;
  const int64_t nblocks = all_blocks + (split ? a.layout->n_tiles[SPANS] * span_blocks : 0);
  const int split_at = split ? (int)all_blocks : 0;
  if (nblocks == 0) return PG_OK;
  dim3 grid((unsigned)nblocks), block(kRopeThreads);
  const pg_kernel kid = inverse ? PG_KERNEL_ROPE_BWD : PG_KERNEL_ROPE;
  prof_begin(kid, a.stream);
  if (a.dtype == PG_F32) {
    rope_kernel<float, float><<<grid, block, 0, a.stream>>>(
        static_cast<const float*>(x0), static_cast<float*>(y0), heads0,
        static_cast<const float*>(x1), static_cast<float*>(y1), heads1, a.d, T, tpb, spans, span_blocks, split_at, tpb1, pos,
        f, rope, sgn, table_out, table_in);
  } else if (in_fp32) {
    rope_kernel<float, __nv_bfloat16><<<grid, block, 0, a.stream>>>(
        static_cast<const float*>(x0), static_cast<__nv_bfloat16*>(y0), heads0,
        static_cast<const float*>(x1), static_cast<__nv_bfloat16*>(y1), heads1, a.d, T, tpb, spans, span_blocks,
        split_at, tpb1, pos, f, rope, sgn, table_out, table_in);
  } else {
    rope_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, block, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(x0), static_cast<__nv_bfloat16*>(y0), heads0,
        static_cast<const __nv_bfloat16*>(x1), static_cast<__nv_bfloat16*>(y1), heads1, a.d, T, tpb,
        spans, span_blocks, split_at, tpb1, pos, f, rope, sgn, table_out, table_in);
  }
  prof_end(kid, a.stream);
  return cuda_check(cudaGetLastError(), "rope launch");
}

// Padded layouts: one block per padding row (grid-stride), 16-byte zero stores over each tensor's
// row, and lse = +inf for every head.
__global__ void __launch_bounds__(256)
pad_fill_kernel(const int32_t* __restrict__ rows, int64_t n, uint4* __restrict__ x0,
                int64_t v0, uint4* __restrict__ x1, int64_t v1, uint4* __restrict__ x2,
                int64_t v2, float* __restrict__ lse, int Hq, int64_t Ttot) {
  for (int64_t i = blockIdx.x; i < n; i += gridDim.x) {
    const int64_t r = rows[i];
    if (r < 0 || r >= Ttot) {
      report(PG_ERR_DEVICE);
      continue;
    }
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t e = threadIdx.x; e < v0; e += blockDim.x) x0[r * v0 + e] = z;
    if (x1)
      for (int64_t e = threadIdx.x; e < v1; e += blockDim.x) x1[r * v1 + e] = z;
    if (x2)
      for (int64_t e = threadIdx.x; e < v2; e += blockDim.x) x2[r * v2 + e] = z;
    if (lse)
      for (int h = threadIdx.x; h < Hq; h += blockDim.x) lse[(size_t)h * Ttot + r] = INFINITY;
  }
}

pg_status launch_pad_fill(const AttnArgs& a, void* x0, int heads0, void* x1, int heads1, void* x2,
                          int heads2, float* lse) {
  const pg_layout* L = a.layout;
  if (L->n_pad_rows == 0) return PG_OK;
  const int64_t es = a.dtype == PG_F32 ? 4 : 2;
  const int32_t* rows = reinterpret_cast<const int32_t*>(static_cast<const char*>(L->tables) +
                                                         L->off_pad_rows);
  const unsigned grid = (unsigned)std::min<int64_t>(L->n_pad_rows, 152 * 8);
  prof_begin(PG_KERNEL_PAD_FILL, a.stream);
  pad_fill_kernel<<<grid, 256, 0, a.stream>>>(
      rows, L->n_pad_rows, static_cast<uint4*>(x0), heads0 * a.d * es / 16,
      static_cast<uint4*>(x1), heads1 * a.d * es / 16, static_cast<uint4*>(x2),
      heads2 * a.d * es / 16, lse, a.Hq, L->total_tokens);
  prof_end(PG_KERNEL_PAD_FILL, a.stream);
  return cuda_check(cudaGetLastError(), "pad fill launch");
}

pg_status launch_fwd_simt(const AttnArgs& a, const void* q, const void* k, const void* v, void* o,
                          float* lse) {
  if (a.dtype == PG_F32)
    return a.d == 64 ? fwd_simt_t<float, 64>(a, q, k, v, o, lse)
                     : fwd_simt_t<float, 128>(a, q, k, v, o, lse);
  return a.d == 64 ? fwd_simt_t<__nv_bfloat16, 64>(a, q, k, v, o, lse)
                   : fwd_simt_t<__nv_bfloat16, 128>(a, q, k, v, o, lse);
}

pg_status launch_bwd_preprocess(const AttnArgs& a, const void* o, const void* dO, const float* lse,
                                float* Dbuf, float* lse2, float* dq_acc, bool lse2_ready) {
  const int T = (int)a.layout->total_tokens;
  const int ldd = (int)padded_tokens(a.layout);
  const size_t threads = (size_t)ldd * a.Hq * (a.d / 8);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  prof_begin(PG_KERNEL_BWD_PREPROCESS, a.stream);
  if (a.dtype == PG_F32)
    bwd_pre_kernel<float><<<blocks, 256, 0, a.stream>>>(
        static_cast<const float*>(o), static_cast<const float*>(dO), lse, Dbuf, lse2, dq_acc,
        a.Hq, a.d, T, ldd, lse2_ready ? 1 : 0);
  else
    bwd_pre_kernel<__nv_bfloat16><<<blocks, 256, 0, a.stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), lse, Dbuf,
        lse2, dq_acc, a.Hq, a.d, T, ldd, lse2_ready ? 1 : 0);
  prof_end(PG_KERNEL_BWD_PREPROCESS, a.stream);
  return cuda_check(cudaGetLastError(), "bwd preprocess launch");
}

pg_status launch_bwd_simt(const AttnArgs& a, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* dO, float* Dbuf,
                          float* dq_acc, float* dk_acc, void* dv) {
  (void)o;
  if (a.dtype == PG_F32)
    return a.d == 64 ? bwd_simt_t<float, 64>(a, q, k, v, dO, lse, Dbuf, dq_acc, dk_acc, dv)
                     : bwd_simt_t<float, 128>(a, q, k, v, dO, lse, Dbuf, dq_acc, dk_acc, dv);
  return a.d == 64
             ? bwd_simt_t<__nv_bfloat16, 64>(a, q, k, v, dO, lse, Dbuf, dq_acc, dk_acc, dv)
             : bwd_simt_t<__nv_bfloat16, 128>(a, q, k, v, dO, lse, Dbuf, dq_acc, dk_acc, dv);
}

pg_status read_status_simt(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_simt, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_simt, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}


}  // namespace pg
