// Grouped-attention backward on the 5th-generation tensor cores (bf16, head_dim 128).
//
// Key-major: one CTA owns 128 keys of one group and one key/value head (a BwdTile) and sweeps, in
// a fixed order, every block of 64 query rows that can see its keys and, for each block, every
// query head of that KV head (the heads innermost, so consecutive steps read neighbouring rows).
// For a prefix key block that is the rest of the prefix and then all responses of the
// group, so the prefix dK / dV -- the sum over the G baseline copies of the shared prefix (Pith
// review of Prefix Grouper, Appendix A.1 objection: the shared prefix's gradient equals the sum of
// the copies' gradients) -- is accumulated in TMEM by one CTA in a fixed order: bitwise
// reproducible, no atomics.  dQ is accumulated across key blocks by TMA reduce-adds into an fp32
// buffer (its summation order is not fixed).
//
// Per query block (64 rows), with K, V resident in shared memory and Q, dO, the blocks' LSE (log2
// units), rowsum(dO * O) and visibility entries arriving by TMA in a 3-stage ring:
//   S^T  = K Q^T          M 128 keys x N 64 queries x K 128   (TMEM cols [0, 64))
//   dP^T = V dO^T         M 128 x N 64 x K 128                 (TMEM cols [64, 128))
//   P^T  = exp2(S^T * scale * log2 e - LSE_2[q]),  dS^T = P^T * (dP^T - Dsum[q])   (registers,
//          one thread per key row, rounded to bf16 and stored into TMEM cols [192, 224) and
//          [224, 256); dS^T also into shared memory, the B operand of dQ^T)
//   dV  += P^T dO         M 128 x N 128 dims x K 64, A = P^T from TMEM  (TMEM cols [256, 384))
//   dK  += dS^T Q         M 128 x N 128 x K 64, A = dS^T from TMEM      (TMEM cols [384, 512))
//   dQ^T = K^T dS^T       M 128 dims x N 64 queries x K 128    (TMEM cols [128, 192)),
//          drained by four warps (one thread per head-dim lane): the warps stage the block, 32
//          query rows at a time, into a shared [32 x 128] fp32 box (each warp its 32 head dims;
//          two boxes alternate) and one thread adds each box into the global dQ accumulator with
//          a TMA bulk reduce-add -- one 16 KB operation per half block, which the memory system
//          takes faster than four 4 KB ones.
// Two threads issue the MMAs: one the score products S^T / dP^T, the other the gradient products
// dV, dK (and dQ^T) of each block as soon as its P^T / dS^T are ready, so the next block's scores
// never queue behind the previous block's gradient waits and the tensor core computes them while
// the softmax warps work on the current ones.
// The epilogue stages dV (bf16) and scale * dK (fp32) row by row in the freed Q / dO rings, then
// each warp writes whole rows: dK rotated back by the inverse RoPE angle (the pair (k, k + d/2)
// of one row; cos/sin from the table the RoPE pass of the same call wrote), coalesced stores.
//
// Warps: 0 TMA producer, 1 TMEM allocation and the score MMAs, 2..9 softmax (key rows; two
// warpgroups split the 64 query columns), 10..13 dQ drain, 14 the gradient MMAs.  Every mbarrier
// wait is bounded.
//
// Instantiated twice: with dQ as above, and without it (kDQ = false: no dQ^T product, no dS^T in
// shared memory, no drain warps; warp 10 issues the gradient MMAs) for the deterministic
// backward, whose dQ comes from the query-major kernel in pg_attn_dq_sm100.cu.
#include <limits.h>
#include <math.h>
#include <string.h>

#include "pg_internal.h"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;

namespace {

constexpr int D = 128;
constexpr int BKV = 128;        // keys per CTA
constexpr int BQ = 64;          // query rows per block
constexpr int NSQ = 3;          // Q / dO stages
constexpr uint32_t KHALF = BKV * 64 * 2;   // 16 KiB: [128 rows][64 cols] bf16
constexpr uint32_t QHALF = BQ * 64 * 2;    // 8 KiB:  [64 rows][64 cols] bf16
// With dQ: warps 10..13 drain dQ and warp 14 issues the gradient MMAs (dV, dK, dQ^T).  Without:
// warp 10 issues them (dV, dK).
constexpr int nthreads(bool with_dq) { return with_dq ? 480 : 352; }
constexpr int grad_warp(bool with_dq) { return with_dq ? 14 : 10; }
constexpr float kLog2e = 1.4426950408889634f;

__device__ int s_status_bwd = 0;

struct BwdSmem {
  uint8_t k[2 * KHALF];
  uint8_t v[2 * KHALF];
  uint8_t q[NSQ][2 * QHALF];
  uint8_t dO[NSQ][2 * QHALF];
  uint8_t ds[KHALF];        // dS^T [128 keys][64 queries] bf16, SW128
  alignas(1024) float dqs[2][BQ / 2][D];    // dQ staging: two [32 queries][128 dims] fp32 boxes
  alignas(128) float lse2[NSQ][BQ];
  alignas(128) float dsum[NSQ][BQ];
  alignas(128) int4 tokq[NSQ][BQ];   // per-token {g0, pe, own_lo, pos} of the block's queries
  uint64_t kv_full;
  uint64_t qd_full[NSQ], qd_empty[NSQ];
  uint64_t s_full, s_free, p_full, pds_free, dq_full, dq_free, mma_done, mma_done2;
  uint32_t tmem;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fail(int code) { atomicCAS(&s_status_bwd, 0, code); }

template <bool kDQ>
__global__ void __launch_bounds__(nthreads(kDQ), 1)
attn_bwd_sm100_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                      const __grid_constant__ CUtensorMap tl2, const __grid_constant__ CUtensorMap tds,
                      const __grid_constant__ CUtensorMap ttok,
                      const __grid_constant__ CUtensorMap tdq, __nv_bfloat16* __restrict__ dk,
                      __nv_bfloat16* __restrict__ dv, const int4* __restrict__ tok,
                      const BwdTile* __restrict__ tiles, int Hq, int Hkv, int Ttot,
                      float scale_log2, float scale, const float2* __restrict__ rope_tab,
                      int hc, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  BwdSmem& sm = *reinterpret_cast<BwdSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tile_id, kh;
  chunked_order(blockIdx.x, gridDim.x / Hkv, Hkv, hc, tile_id, kh);
  const BwdTile tl = tiles[tile_id];
  if (tl.k0 < 0 || tl.k1 > Ttot || tl.k0 >= tl.k1 || tl.k1 - tl.k0 > BKV || tl.q_lo < 0 ||
      tl.q_hi > Ttot || tl.q_lo >= tl.q_hi) {
    if (threadIdx.x == 0) fail(PG_ERR_DEVICE);
    return;
  }
  const int rep = Hq / Hkv;
  // Query blocks start at a multiple of 4 rows (16-byte aligned TMA coordinates for the fp32
  // rows); the few rows before q_lo that this adds never see the block's keys (they are masked).
  const int qt0 = tl.q_lo & ~3;
  const int nqt = (tl.q_hi - qt0 + BQ - 1) / BQ;
  const int n_it = rep * nqt;

  if (threadIdx.x == 0) {
    mbar_init(&sm.kv_full, 1);
    for (int s = 0; s < NSQ; ++s) {
      mbar_init(&sm.qd_full[s], 1);
      mbar_init(&sm.qd_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, 256);
    mbar_init(&sm.p_full, 256);
    mbar_init(&sm.pds_free, 1);
    mbar_init(&sm.dq_full, 1);
    mbar_init(&sm.dq_free, 128);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.mma_done2, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t t_s = tmem, t_dp = tmem + 64, t_dq = tmem + 128, t_p = tmem + 192,
                 t_ds = tmem + 224, t_dv = tmem + 256, t_dk = tmem + 384;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer ---------
    const bool leader = elect_one();
    if (leader) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tl2);
      prefetch_tmap(&tds);
      prefetch_tmap(&ttok);
      mbar_expect_tx(&sm.kv_full, 4 * KHALF);
      tma_load_2d(sm.k, &tk, &sm.kv_full, kh * D, tl.k0);
      tma_load_2d(sm.k + KHALF, &tk, &sm.kv_full, kh * D + 64, tl.k0);
      tma_load_2d(sm.v, &tv, &sm.kv_full, kh * D, tl.k0);
      tma_load_2d(sm.v + KHALF, &tv, &sm.kv_full, kh * D + 64, tl.k0);
    }
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSQ;
      const int h = kh * rep + it % rep;
      const int qt = qt0 + (it / rep) * BQ;
      if (!warp_wait(&sm.qd_empty[st], ((it / NSQ) & 1) ^ 1, wait_ns)) { ok = false; break; }
      if (leader) {
        mbar_expect_tx(&sm.qd_full[st], 4 * QHALF + 2 * BQ * 4 + BQ * 16);
        tma_load_2d(sm.q[st], &tq, &sm.qd_full[st], h * D, qt);
        tma_load_2d(sm.q[st] + QHALF, &tq, &sm.qd_full[st], h * D + 64, qt);
        tma_load_2d(sm.dO[st], &tdo, &sm.qd_full[st], h * D, qt);
        tma_load_2d(sm.dO[st] + QHALF, &tdo, &sm.qd_full[st], h * D + 64, qt);
        tma_load_2d(sm.lse2[st], &tl2, &sm.qd_full[st], qt, h);
        tma_load_2d(sm.dsum[st], &tds, &sm.qd_full[st], qt, h);
        tma_load_2d(sm.tokq[st], &ttok, &sm.qd_full[st], 0, qt);
      }
      __syncwarp();
      ++issued;
    }
    if (!ok && lane == 0) fail(PG_ERR_TIMEOUT);
    if (leader) {
      mbar_wait(&sm.kv_full, 0, wait_ns);
      for (int it = (issued > NSQ ? issued - NSQ : 0); it < issued; ++it)
        mbar_wait(&sm.qd_full[it % NSQ], (it / NSQ) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ score MMAs -------
    if (elect_one()) {
      constexpr uint32_t id_s = idesc_bf16(BKV, BQ, 0, 0);     // S^T, dP^T
      // Descriptor bases (K-major operands: LBO unused).
      const uint64_t kd = sdesc_sw128(smem_u32(sm.k), 16, 1024);
      const uint64_t vd = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t dod0 = sdesc_sw128(smem_u32(sm.dO[0]), 16, 1024);
      bool ok = mbar_wait(&sm.kv_full, 0, wait_ns);
      for (int it = 0; ok && it < n_it; ++it) {
        const int st = it % NSQ;
        if (!mbar_wait(&sm.qd_full[st], (it / NSQ) & 1, wait_ns)) { ok = false; break; }
        if (it > 0 && !mbar_wait(&sm.s_free, (it - 1) & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint64_t qd = desc_add(qd0, st * 2 * QHALF), dod = desc_add(dod0, st * 2 * QHALF);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * KHALF + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * QHALF + (kk & 3) * 32;
          mma_ss(t_s, desc_add(kd, ko), desc_add(qd, qo), id_s, kk != 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk >> 2) * KHALF + (kk & 3) * 32;
          const uint32_t qo = (kk >> 2) * QHALF + (kk & 3) * 32;
          mma_ss(t_dp, desc_add(vd, ko), desc_add(dod, qo), id_s, kk != 0);
        }
        mma_commit(&sm.s_full);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------------------------------------ softmax (keys) ----
    // Two warpgroups: warps 2..5 take query columns 0..31 of the block, warps 6..9 columns
    // 32..63; warp w reads TMEM lanes 32 * (w % 4) .. + 31 (its key rows).
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quarter * 32 + lane;
    const int key = tl.k0 + r;
    const bool kvalid = key < tl.k1;
    const int keyc = kvalid ? key : tl.k1 - 1;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int c0 = half * 32;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it % NSQ;
      const int qt = qt0 + (it / rep) * BQ;
      if (!warp_wait(&sm.s_full, it & 1, wait_ns)) { ok = false; break; }
      if (!warp_wait(&sm.qd_full[st], (it / NSQ) & 1, wait_ns)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[32], dr[32];
      tmem_ld32(t_s + lane_addr + c0, sr);
      tmem_ld32(t_dp + lane_addr + c0, dr);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.s_free);
      const bool full = (qt >= tl.k0 + BKV - 1) && (tl.k1 - tl.k0 == BKV) && (tl.k1 <= tl.pe) &&
                        (qt + BQ <= tl.q_hi);
      const float4* l2v = reinterpret_cast<const float4*>(sm.lse2[st] + c0);
      const float4* dsv = reinterpret_cast<const float4*>(sm.dsum[st] + c0);
      uint32_t pw[16], dw[16];
      if (full) {
        // Column pairs through the packed fp32 unit (same roundings as the scalar forms).
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l = l2v[c4], dd = dsv[c4];
          float p0, p1, p2, p3, d0, d1, d2, d3;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * c4]), __uint_as_float(sr[4 * c4 + 1])),
                           sc2, f2_pack(-l.x, -l.y)), p0, p1);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3])),
                           sc2, f2_pack(-l.z, -l.w)), p2, p3);
          p0 = fast_exp2(p0);
          p1 = fast_exp2(p1);
          p2 = fast_exp2(p2);
          p3 = fast_exp2(p3);
          pw[2 * c4] = pack_bf16x2(p0, p1);
          pw[2 * c4 + 1] = pack_bf16x2(p2, p3);
          f2_unpack(f2_mul(f2_pack(p0, p1),
                           f2_sub(f2_pack(__uint_as_float(dr[4 * c4]), __uint_as_float(dr[4 * c4 + 1])),
                                  f2_pack(dd.x, dd.y))), d0, d1);
          f2_unpack(f2_mul(f2_pack(p2, p3),
                           f2_sub(f2_pack(__uint_as_float(dr[4 * c4 + 2]), __uint_as_float(dr[4 * c4 + 3])),
                                  f2_pack(dd.z, dd.w))), d2, d3);
          dw[2 * c4] = pack_bf16x2(d0, d1);
          dw[2 * c4 + 1] = pack_bf16x2(d2, d3);
        }
      } else {
        const int4* tq4 = sm.tokq[st] + c0;
        const float* l2 = sm.lse2[st] + c0;
        const float* ds_ = sm.dsum[st] + c0;
        // Branch-free visibility (bitwise, not short-circuit, so the unrolled loop stays
        // straight-line): query t sees this key iff key <= t < q_hi and the key is a prefix key or
        // lies in t's own response.  An invisible entry's exponent is -inf, so P = 0 and dS = 0.
        const bool prefix_key = keyc < tl.pe;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int t0 = qt + c0 + c, t1 = t0 + 1;
          const bool v0 = kvalid & (t0 < tl.q_hi) & (keyc <= t0) & (prefix_key | (keyc >= tq4[c].z));
          const bool v1 =
              kvalid & (t1 < tl.q_hi) & (keyc <= t1) & (prefix_key | (keyc >= tq4[c + 1].z));
          const float a0 = fmaf(__uint_as_float(sr[c]), scale_log2, -l2[c]);
          const float a1 = fmaf(__uint_as_float(sr[c + 1]), scale_log2, -l2[c + 1]);
          const float p0 = fast_exp2(v0 ? a0 : -INFINITY);
          const float p1 = fast_exp2(v1 ? a1 : -INFINITY);
          pw[c >> 1] = pack_bf16x2(p0, p1);
          dw[c >> 1] = pack_bf16x2(p0 * (__uint_as_float(dr[c]) - ds_[c]),
                                   p1 * (__uint_as_float(dr[c + 1]) - ds_[c + 1]));
        }
      }
      // The previous block's gradient products must be done with P^T / dS^T.
      if (it > 0 && !warp_wait(&sm.pds_free, (it - 1) & 1, wait_ns)) { ok = false; break; }
      tc_fence_after();
      tmem_st16(t_p + half * 16 + lane_addr, pw);
      tmem_st16(t_ds + half * 16 + lane_addr, dw);
      if constexpr (kDQ) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const uint32_t off = sw128_offset(r, half * 4 + ch);
          *reinterpret_cast<uint4*>(sm.ds + off) =
              make_uint4(dw[4 * ch], dw[4 * ch + 1], dw[4 * ch + 2], dw[4 * ch + 3]);
        }
      }
      tmem_st_wait();
      if constexpr (kDQ) fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sm.p_full);
    }
    // Epilogue, through shared memory (the Q / dO rings, 96 KB, are free once every product has
    // completed): each thread stages its key row -- dV rounded to bf16 (256-byte rows), scale * dK
    // in fp32 (512-byte rows), 16-byte chunks XOR-swizzled by the row so the staging stores are
    // conflict-free -- then each warp writes whole rows, so the global stores and the RoPE table
    // reads are coalesced instead of every warp access touching 32 rows.  dK is rotated back by
    // the key's RoPE angle on the way out: columns p and p + 64 form rotation pair p, and lane l
    // of a warp handles pairs 2l and 2l + 1 of a row.  The warp's 16 rows of (cos, sin) are read
    // into registers before the wait for the last products, so their L2 round trip (long under
    // the dQ reduce traffic of the other CTAs) overlaps it and the staging.  The eight warps
    // decide together, so none waits at the staging barrier alone.
    const int wl = warp - 2;                    // rows 16 wl .. 16 wl + 15 in the copy-out
    const int nrows = tl.k1 - tl.k0;
    float4 cs[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int row = wl * 16 + i;
      cs[i] = (rope_tab && row < nrows)
                  ? *reinterpret_cast<const float4*>(rope_tab + (size_t)(tl.k0 + row) * (D / 2) +
                                                     2 * lane)
                  : make_float4(1.f, 0.f, 1.f, 0.f);
    }
    if (named_bar_and(2, 256, ok && warp_wait(&sm.pds_free, (n_it - 1) & 1, wait_ns))) {
      tc_fence_after();
      uint8_t* dks = sm.q[0];                   // [128][128] fp32
      uint8_t* dvs = sm.q[0] + BKV * D * 4;     // [128][128] bf16
      if (half == 0) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v32[32];
          tmem_ld32(t_dv + lane_addr + c * 32, v32);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t* e = v32 + 8 * k;
            *reinterpret_cast<uint4*>(dvs + stage_offset(r, c * 4 + k, 256)) = make_uint4(
                pack_bf16x2(__uint_as_float(e[0]), __uint_as_float(e[1])),
                pack_bf16x2(__uint_as_float(e[2]), __uint_as_float(e[3])),
                pack_bf16x2(__uint_as_float(e[4]), __uint_as_float(e[5])),
                pack_bf16x2(__uint_as_float(e[6]), __uint_as_float(e[7])));
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t a32[32];
          tmem_ld32(t_dk + lane_addr + c * 32, a32);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint32_t* e = a32 + 4 * k;
            *reinterpret_cast<float4*>(dks + stage_offset(r, c * 8 + k, 512)) =
                make_float4(__uint_as_float(e[0]) * scale, __uint_as_float(e[1]) * scale,
                            __uint_as_float(e[2]) * scale, __uint_as_float(e[3]) * scale);
          }
        }
      }
      named_bar_sync(2, 256);
#pragma unroll 4
      for (int i = 0; i < 8; ++i) {             // dV: two rows per access, 16 lanes x 16 B each
        const int row = wl * 16 + 2 * i + (lane >> 4), ch = lane & 15;
        if (row < nrows)
          *reinterpret_cast<uint4*>(dv + ((size_t)(tl.k0 + row) * Hkv + kh) * D + ch * 8) =
              *reinterpret_cast<const uint4*>(dvs + stage_offset(row, ch, 256));
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {            // dK: one row per access
        const int row = wl * 16 + i;
        if (row < nrows) {
          const float2 x1 = *reinterpret_cast<const float2*>(
              dks + stage_offset(row, lane >> 1, 512) + (lane & 1) * 8);
          const float2 x2 = *reinterpret_cast<const float2*>(
              dks + stage_offset(row, 16 + (lane >> 1), 512) + (lane & 1) * 8);
          float lo0 = x1.x, lo1 = x1.y, hi0 = x2.x, hi1 = x2.y;
          if (rope_tab) {
            const float4 e = cs[i];             // (cos, sin) of pairs 2l and 2l + 1
            lo0 = x1.x * e.x + x2.x * e.y;
            hi0 = x2.x * e.x - x1.x * e.y;
            lo1 = x1.y * e.z + x2.y * e.w;
            hi1 = x2.y * e.z - x1.y * e.w;
          }
          __nv_bfloat16* drow = dk + ((size_t)(tl.k0 + row) * Hkv + kh) * D;
          *reinterpret_cast<uint32_t*>(drow + 2 * lane) = pack_bf16x2(lo0, lo1);
          *reinterpret_cast<uint32_t*>(drow + 64 + 2 * lane) = pack_bf16x2(hi0, hi1);
        }
      }
    } else {
      ok = false;
    }
    if (!ok) fail(PG_ERR_TIMEOUT);
  } else if (warp == grad_warp(kDQ)) {
    // ------------------------------------------------------------------ gradient MMAs ----
    // Second issuing thread: dV += P^T dO and dK += dS^T Q of each block as soon as its P^T /
    // dS^T are in TMEM, then (with dQ) dQ^T = K^T dS^T once the drain warps have read the
    // previous block's dQ^T.  Block j's S^T / dP^T products completed before its softmax could
    // signal p_full, so the qd_empty commit below covers every reader of the stage.
    if (elect_one()) {
      constexpr uint32_t id_g = idesc_bf16(BKV, D, 0, 1);      // dV, dK
      constexpr uint32_t id_q = idesc_bf16(D, BQ, 1, 1);       // dQ^T
      // MN-major operands: LBO = the 64-column half.
      const uint64_t qmn0 = sdesc_sw128(smem_u32(sm.q[0]), QHALF, 1024);
      const uint64_t domn0 = sdesc_sw128(smem_u32(sm.dO[0]), QHALF, 1024);
      const uint64_t kmn = sdesc_sw128(smem_u32(sm.k), KHALF, 1024);
      const uint64_t dsmn = sdesc_sw128(smem_u32(sm.ds), QHALF, 1024);
      bool ok = true;
      for (int jp = 0; jp < n_it; ++jp) {
        const int sp = jp % NSQ;
        if (!mbar_wait(&sm.p_full, jp & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint64_t qmn = desc_add(qmn0, sp * 2 * QHALF);
        const uint64_t domn = desc_add(domn0, sp * 2 * QHALF);
        const uint32_t acc0 = jp != 0;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(t_dv, t_p + kk * 8, desc_add(domn, kk * 2048), id_g, kk == 0 ? acc0 : 1u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(t_dk, t_ds + kk * 8, desc_add(qmn, kk * 2048), id_g, kk == 0 ? acc0 : 1u);
        mma_commit(&sm.qd_empty[sp]);
        if constexpr (kDQ) {
          if (jp >= 1 && !mbar_wait(&sm.dq_free, (jp - 1) & 1, wait_ns)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_ss(t_dq, desc_add(kmn, kk * 2048), desc_add(dsmn, kk * 2048), id_q, kk != 0);
          mma_commit(&sm.dq_full);
        } else {
          (void)kmn;
          (void)dsmn;
          (void)id_q;
        }
        mma_commit(&sm.pds_free);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.mma_done2);
      mbar_wait(&sm.mma_done2, 0, wait_ns);
    }
    __syncwarp();
  } else if (kDQ) {
    // ------------------------------------------------------------------ dQ drain ---------
    const int quarter = warp & 3;                  // this warp's 32 head dims (= TMEM lanes)
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    // One thread issues the reduce-adds of all four warps: a whole [32 x 128] box per half
    // block (fewer, larger bulk operations than one per warp).
    const bool issuer = warp == 10 && lane == 0;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int h = kh * rep + it % rep;
      const int qt = qt0 + (it / rep) * BQ;
      // The four drain warps leave the loop together, so none waits at a barrier below alone.
      if (!named_bar_and(1, 128, warp_wait(&sm.dq_full, it & 1, wait_ns))) { ok = false; break; }
      tc_fence_after();
      uint32_t g[64];
      tmem_ld32(t_dq + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(&g[0]));
      tmem_ld32(t_dq + lane_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&g[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.dq_free);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float (*box)[D] = sm.dqs[hf];
        // The reduce that last read this box (the previous block's) must be done with it; the
        // other box's may still be reading.
        if (issuer) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        named_bar_sync(1, 128);
#pragma unroll
        for (int c = 0; c < BQ / 2; ++c)
          box[c][quarter * 32 + lane] = __uint_as_float(g[hf * (BQ / 2) + c]) * scale;
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (issuer) {
          // Rows past the group receive +0; rows past the tensor are clipped by the TMA unit.
          tma_reduce_add_2d(&tdq, &box[0][0], h * D, qt + hf * (BQ / 2));
          bulk_commit_group();
        }
      }
    }
    if (issuer) bulk_wait_group0();
    __syncwarp();
    if (!ok) fail(PG_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool bwd_sm100_supported(const AttnArgs& a) { return a.dtype == PG_BF16 && a.d == 128; }

pg_status launch_bwd_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse2, const float* Dbuf, float* dq_acc,
                           void* dk, void* dv, const float2* rope_tab) {
  const pg_layout* L = a.layout;
  const int64_t T = L->total_tokens;
  const int64_t Tp = padded_tokens(L);
  CUtensorMap tq, tk, tv, tdo, tl2, tds, ttok, tdq;
  pg_status st = make_tmap_2d_bf16(&tq, q, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 2, 64, BQ);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tdo, dO, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 2, 64, BQ);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tk, k, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BKV);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tv, v, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BKV);
  if (st == PG_OK) st = make_tmap_2d_b32(&tl2, lse2, true, Tp, a.Hq, Tp * 4, BQ, 1);
  if (st == PG_OK) st = make_tmap_2d_b32(&tds, Dbuf, true, Tp, a.Hq, Tp * 4, BQ, 1);
  if (st == PG_OK) st = make_tmap_2d_b32(&ttok, tokens(L), false, 4, T, 16, 4, BQ);
  // Without a dQ accumulator the kernel computes dK and dV only (dQ comes from the query-major
  // kernel); its dQ tensor map is then never read.
  const bool with_dq = dq_acc != nullptr;
  memset(&tdq, 0, sizeof(tdq));
  if (st == PG_OK && with_dq)
    st = make_tmap_2d_b32(&tdq, dq_acc, true, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 4, D,
                          BQ / 2);
  if (st != PG_OK) return st;
  const size_t smem = sizeof(BwdSmem) + 1024;
  auto kern = with_dq ? attn_bwd_sm100_kernel<true> : attn_bwd_sm100_kernel<false>;
  st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem),
                  "bwd smem attribute");
  if (st != PG_OK) return st;
  prof_begin(PG_KERNEL_BWD_DKDV, a.stream);
  kern<<<(unsigned)(L->n_tiles[BWD128] * a.Hkv), nthreads(with_dq), smem, a.stream>>>(
      tq, tk, tv, tdo, tl2, tds, ttok, tdq, static_cast<__nv_bfloat16*>(dk),
      static_cast<__nv_bfloat16*>(dv), tokens(L), tiles<BwdTile>(L, BWD128), a.Hq, a.Hkv, (int)T,
      a.scale * kLog2e, a.scale, rope_tab, order_chunk(a.Hkv, a.Hq / a.Hkv), 2000000000ull);
  prof_end(PG_KERNEL_BWD_DKDV, a.stream);
  return cuda_check(cudaGetLastError(), "bwd sm100 launch");
}

pg_status read_status_bwd_sm100(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_bwd, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_bwd, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}

}  // namespace pg
