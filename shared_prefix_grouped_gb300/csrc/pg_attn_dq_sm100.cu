// Query-major dQ of grouped attention on the 5th-generation tensor cores (bf16, head_dim 128):
// the deterministic half of the backward.
//
// A CTA owns 128 packed query rows of one group and one query head (a 128-row FwdTile) and streams
// the same 128-key K/V tiles the forward visits for those rows: the group's prefix, then the
// responses' part (Pith review of Prefix Grouper, "What carries the argument": a response row sees
// the whole prefix and its own response).  With LSE and rowsum(dO * O) of its rows known from the
// forward and the preprocess, each key tile gives
//   S  = Q K^T            M 128 rows x N 128 keys x K 128    (TMEM cols [0, 128))
//   dP = dO V^T           M 128 x N 128 x K 128              (TMEM cols [128, 256))
//   P  = exp2(S * scale * log2 e - LSE_2),  dS = P * (dP - Dsum)     (registers; dS rounded to
//        bf16 and stored into TMEM cols [384 + 64 b, ...), double-buffered, as the A operand of)
//   dQ += dS K            M 128 x N 128 dims x K 128 keys, K as the MN-major B operand
//                                                            (TMEM cols [256, 384))
// and the epilogue applies the softmax scale, stages dQ in the freed Q / dO tiles, and writes it
// in bf16 by whole rows, rotated back by the inverse RoPE angle (the pair (k, k + d/2) of a row;
// cos/sin from the table the RoPE pass of the same call wrote).  Every row's dQ is summed by one CTA over the keys in a fixed
// order: no atomics, bitwise reproducible.
//
// Warps (352 threads): 0 TMA producer (Q and dO once, K and V tiles into a 2-stage ring), 1 TMEM
// allocation and the S / dP MMAs, 10 the dQ MMAs (a second issuing thread, so dQ of tile j never
// waits behind the next tile's loads or score products), 2..9 softmax and epilogue (warp w reads
// TMEM lanes 32 (w % 4) .. + 31; warps 2..5 take key columns 0..63, warps 6..9 columns 64..127).
// Every mbarrier wait is bounded (PG_ERR_TIMEOUT in the status word, then an orderly exit).
#include <math.h>

#include "pg_internal.h"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;

namespace {

constexpr int D = 128;
constexpr int BM = 128;                   // query rows per CTA
constexpr int BN = 128;                   // keys per tile
constexpr int NS = 2;                     // K/V stages
constexpr uint32_t QH = BM * 64 * 2;      // [128 rows][64 dims] bf16: 16 KiB
constexpr uint32_t KH = BN * 64 * 2;      // [128 keys][64 dims] bf16: 16 KiB
constexpr int NTHREADS = 352;
constexpr float kLog2e = 1.4426950408889634f;

__device__ int s_status_dq = 0;

// Key tile j of the CTA: the tiles of its causal key ranges first, then of its own range.
// Built once per CTA in shared memory.
struct Plan {
  int n_r, n_a, n;
  int lo[kMaxKeyRanges], hi[kMaxKeyRanges], cum[kMaxKeyRanges + 1];
  __device__ void init(const FwdTile& t, const int2* ivs) {
    KeyRanges kr;
    kr.init(t, ivs);
    n_r = kr.n;
    cum[0] = 0;
    n_a = 0;
    for (int r = 0; r < kr.n; ++r) {
      lo[r] = kr.lo[r];
      hi[r] = kr.hi[r];
      cum[r + 1] = cum[r] + (hi[r] - lo[r] + BN - 1) / BN;
      if (r + 1 == kr.n_causal) n_a = cum[r + 1];
    }
    n = cum[kr.n];
  }
};

// Walks the key tiles of a Plan in increasing j, keeping the current range in registers (the
// tables in shared memory are read only when a range ends).
struct TileCursor {
  int r, base, next, lo, hi;
  __device__ explicit TileCursor(const Plan& p) : r(0), base(0), next(p.cum[1]), lo(p.lo[0]), hi(p.hi[0]) {}
  __device__ int seek(const Plan& p, int j) {   // returns the first key of tile j; hi = its range end
    while (j >= next && r + 1 < p.n_r) {
      ++r;
      base = next;
      next = p.cum[r + 1];
      lo = p.lo[r];
      hi = p.hi[r];
    }
    return lo + (j - base) * BN;
  }
};

struct DqSmem {
  uint8_t q[2 * QH];
  uint8_t dO[2 * QH];
  uint8_t k[NS][2 * KH];
  uint8_t v[NS][2 * KH];
  uint64_t q_full;
  uint64_t kv_full[NS], kv_empty[NS];
  uint64_t s_full, s_free, p_full[2], ds_free[2], dq_done, mma_done, mma_done2;
  uint32_t tmem;
  Plan plan;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fail(int code) { atomicCAS(&s_status_dq, 0, code); }

__global__ void __launch_bounds__(NTHREADS, 1)
attn_dq_sm100_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                     const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                     __nv_bfloat16* __restrict__ dq, const float* __restrict__ lse2,
                     const float* __restrict__ dsum, int64_t ldl, const int4* __restrict__ tok,
                     const FwdTile* __restrict__ tiles, const int2* __restrict__ ivs, int Hq,
                     int Hkv, int Ttot,
                     float scale_log2, float scale, const float2* __restrict__ rope_tab,
                     int hc, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  DqSmem& sm = *reinterpret_cast<DqSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tile_id, h;
  chunked_order(blockIdx.x, gridDim.x / Hq, Hq, hc, tile_id, h);
  const int kh = h / (Hq / Hkv);
  const FwdTile tl = tiles[tile_id];
  if (tl.q0 < 0 || tl.q1 > Ttot || tl.q0 >= tl.q1 || tl.q1 - tl.q0 > BM || tl.g0 < 0 ||
      tl.s_hi > Ttot || tl.a_cnt < 0 || tl.a_cnt > kMaxExtraRanges) {
    if (threadIdx.x == 0) fail(PG_ERR_DEVICE);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.kv_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.s_free, 8);      // softmax warps
    mbar_init(&sm.p_full[0], 8);
    mbar_init(&sm.p_full[1], 8);
    mbar_init(&sm.ds_free[0], 1);
    mbar_init(&sm.ds_free[1], 1);
    mbar_init(&sm.dq_done, 1);
    mbar_init(&sm.mma_done, 1);
    mbar_init(&sm.mma_done2, 1);
    fence_mbar_init();
    sm.plan.init(tl, ivs);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dq = tmem + 256, t_ds = tmem + 384;
  const Plan& pl = sm.plan;
  const int n = pl.n, n_a = pl.n_a;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer -----
    if (elect_one()) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tdo);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      const int xq = h * D, xk = kh * D;
      mbar_expect_tx(&sm.q_full, 4 * QH);
      tma_load_2d(sm.q, &tq, &sm.q_full, xq, tl.q0);
      tma_load_2d(sm.q + QH, &tq, &sm.q_full, xq + 64, tl.q0);
      tma_load_2d(sm.dO, &tdo, &sm.q_full, xq, tl.q0);
      tma_load_2d(sm.dO + QH, &tdo, &sm.q_full, xq + 64, tl.q0);
      int issued = 0;
      TileCursor cur(pl);
      for (int j = 0; j < n; ++j) {
        const int s = j % NS;
        if (!mbar_wait(&sm.kv_empty[s], ((j / NS) & 1) ^ 1, wait_ns)) {
          fail(PG_ERR_TIMEOUT);
          break;
        }
        const int kt = cur.seek(pl, j);
        mbar_expect_tx(&sm.kv_full[s], 4 * KH);
        tma_load_2d(sm.k[s], &tk, &sm.kv_full[s], xk, kt);
        tma_load_2d(sm.k[s] + KH, &tk, &sm.kv_full[s], xk + 64, kt);
        tma_load_2d(sm.v[s], &tv, &sm.kv_full[s], xk, kt);
        tma_load_2d(sm.v[s] + KH, &tv, &sm.kv_full[s], xk + 64, kt);
        ++issued;
      }
      // Leave no copy in flight.
      mbar_wait(&sm.q_full, 0, wait_ns);
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
        mbar_wait(&sm.kv_full[j % NS], (j / NS) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S / dP MMAs ------
    if (elect_one()) {
      constexpr uint32_t id_s = idesc_bf16(BM, BN, 0, 0);
      const uint64_t qd = sdesc_sw128(smem_u32(sm.q), 16, 1024);
      const uint64_t dod = sdesc_sw128(smem_u32(sm.dO), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), 16, 1024);
      bool ok = mbar_wait(&sm.q_full, 0, wait_ns);
      for (int j = 0; ok && j < n; ++j) {
        const int s = j % NS;
        if (!mbar_wait(&sm.kv_full[s], (j / NS) & 1, wait_ns)) { ok = false; break; }
        // S and dP are single-buffered: the softmax warps must have read tile j - 1's.
        if (j > 0 && !mbar_wait(&sm.s_free, (j - 1) & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kd = desc_add(kd0, s * 2 * KH), vd = desc_add(vd0, s * 2 * KH);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * QH + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * KH + (kk & 3) * 32;
          mma_ss(t_s, desc_add(qd, qo), desc_add(kd, ko), id_s, kk != 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * QH + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * KH + (kk & 3) * 32;
          mma_ss(t_dp, desc_add(dod, qo), desc_add(vd, ko), id_s, kk != 0);
        }
        mma_commit(&sm.s_full);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------------ dQ MMAs ----------
    // dQ += dS K of tile j once its dS is in TMEM.  Tile j's S / dP products completed before its
    // softmax could signal p_full, so the kv_empty commit covers every reader of the stage.
    if (elect_one()) {
      constexpr uint32_t id_q = idesc_bf16(BM, D, 0, 1);    // K as the MN-major B operand
      const uint64_t kmn0 = sdesc_sw128(smem_u32(sm.k[0]), KH, 1024);
      bool ok = true;
      for (int j = 0; j < n; ++j) {
        const int b = j & 1, s = j % NS;
        // One p_full per dS buffer: tile j + 2 reuses buffer b only after this product read it.
        if (!mbar_wait(&sm.p_full[b], (j >> 1) & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kmn = desc_add(kmn0, s * 2 * KH);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(t_dq, t_ds + 64 * b + kk * 8, desc_add(kmn, kk * 2048), id_q,
                 (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&sm.ds_free[b]);
        mma_commit(&sm.kv_empty[s]);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.dq_done);
      mma_commit(&sm.mma_done2);
      mbar_wait(&sm.mma_done2, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue -
    // (warps 2..9)
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;            // key columns [64 half, 64 half + 64)
    const int r = quarter * 32 + lane;
    const int row = tl.q0 + r;
    const bool valid = row < tl.q1;
    const int rowc = valid ? row : tl.q1 - 1;
    const int4 ti = tok[rowc];                   // {g0, pe, own_lo, pos}
    const float l2r = lse2[(size_t)h * ldl + rowc];
    const float dr_ = dsum[(size_t)h * ldl + rowc];
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    TileCursor cur(pl);
    for (int j = 0; j < n; ++j) {
      const int kt = cur.seek(pl, j);
      const int hi = cur.hi;
      if (!warp_wait(&sm.s_full, j & 1, wait_ns)) { ok = false; break; }
      tc_fence_after();
      // The row's visible keys in this tile: one contiguous run [lo, lo + len) of columns.
      const bool full = (j < n_a) && (kt + BN <= hi) && (kt + BN - 1 <= tl.q0);
      const int lo = (j < n_a) ? 0 : max(ti.z - kt, 0);
      const int len = full ? BN : max(min(hi, rowc + 1) - kt - lo, 0);
      uint32_t dw[32];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int col0 = 64 * half + 32 * c2;
        uint32_t sr[32], dr[32];
        tmem_ld32(t_s + lane_addr + col0, sr);
        tmem_ld32(t_dp + lane_addr + col0, dr);
        tmem_ld_wait();
        if (c2 == 1) {
          tc_fence_before();
          warp_arrive(&sm.s_free);
        }
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const bool v0 = (unsigned)(col0 + e - lo) < (unsigned)len;
          const bool v1 = (unsigned)(col0 + e + 1 - lo) < (unsigned)len;
          const float a0 = fmaf(__uint_as_float(sr[e]), scale_log2, -l2r);
          const float a1 = fmaf(__uint_as_float(sr[e + 1]), scale_log2, -l2r);
          const float p0 = fast_exp2(v0 ? a0 : -INFINITY);
          const float p1 = fast_exp2(v1 ? a1 : -INFINITY);
          dw[16 * c2 + (e >> 1)] = pack_bf16x2(p0 * (__uint_as_float(dr[e]) - dr_),
                                               p1 * (__uint_as_float(dr[e + 1]) - dr_));
        }
      }
      // dS is double-buffered in TMEM: the dQ product that read this buffer two tiles ago must
      // be done.
      const int b = j & 1;
      if (j >= 2 && !warp_wait(&sm.ds_free[b], ((j >> 1) - 1) & 1, wait_ns)) { ok = false; break; }
      tc_fence_after();
      tmem_st32(t_ds + 64 * b + 32 * half + lane_addr, dw);
      tmem_st_wait();
      tc_fence_before();
      warp_arrive(&sm.p_full[b]);
    }
    // Epilogue, through shared memory (the Q and dO tiles, 64 KB, are free once every product has
    // completed): each thread stages scale * dQ of its row's rotation pairs (k, k + 64), k in
    // [32 half, 32 half + 32), in fp32 (512-byte rows, 16-byte chunks XOR-swizzled by the row so
    // the staging stores are conflict-free); then each warp writes whole rows, rotated back by the
    // row's RoPE angle -- lane l handles pairs 2l and 2l + 1 -- so the global stores and the table
    // reads are coalesced instead of every warp access touching 32 rows.  The warp's 16 rows of
    // (cos, sin) are read before the wait for the last dQ product, whose L2 round trip they then
    // overlap.  The eight warps decide together, so none waits at the staging barrier alone.
    const int wl = warp - 2;                    // rows 16 wl .. 16 wl + 15 in the copy-out
    const int nrows = tl.q1 - tl.q0;
    float4 cs[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rr = wl * 16 + i;
      cs[i] = (rope_tab && rr < nrows)
                  ? *reinterpret_cast<const float4*>(rope_tab + (size_t)(tl.q0 + rr) * (D / 2) +
                                                     2 * lane)
                  : make_float4(1.f, 0.f, 1.f, 0.f);
    }
    if (named_bar_and(2, 256, ok && warp_wait(&sm.dq_done, 0, wait_ns))) {
      tc_fence_after();
      uint8_t* dqs = sm.q;                      // [128][128] fp32 over the Q and dO tiles
#pragma unroll
      for (int part = 0; part < 2; ++part) {    // columns 32 half + 64 part .. + 31
        uint32_t a32[32];
        tmem_ld32(t_dq + lane_addr + 64 * part + 32 * half, a32);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t* e = a32 + 4 * k;
          *reinterpret_cast<float4*>(dqs + stage_offset(r, 16 * part + 8 * half + k, 512)) =
              make_float4(__uint_as_float(e[0]) * scale, __uint_as_float(e[1]) * scale,
                          __uint_as_float(e[2]) * scale, __uint_as_float(e[3]) * scale);
        }
      }
      named_bar_sync(2, 256);
#pragma unroll
      for (int i = 0; i < 16; ++i) {            // one row per access
        const int rr = wl * 16 + i;
        if (rr < nrows) {
          const float2 x1 = *reinterpret_cast<const float2*>(
              dqs + stage_offset(rr, lane >> 1, 512) + (lane & 1) * 8);
          const float2 x2 = *reinterpret_cast<const float2*>(
              dqs + stage_offset(rr, 16 + (lane >> 1), 512) + (lane & 1) * 8);
          float lo0 = x1.x, lo1 = x1.y, hi0 = x2.x, hi1 = x2.y;
          if (rope_tab) {
            const float4 e = cs[i];             // (cos, sin) of pairs 2l and 2l + 1
            lo0 = x1.x * e.x + x2.x * e.y;
            hi0 = x2.x * e.x - x1.x * e.y;
            lo1 = x1.y * e.z + x2.y * e.w;
            hi1 = x2.y * e.z - x1.y * e.w;
          }
          __nv_bfloat16* out = dq + ((size_t)(tl.q0 + rr) * Hq + h) * D;
          *reinterpret_cast<uint32_t*>(out + 2 * lane) = pack_bf16x2(lo0, lo1);
          *reinterpret_cast<uint32_t*>(out + 64 + 2 * lane) = pack_bf16x2(hi0, hi1);
        }
      }
    } else {
      ok = false;
    }
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

bool dq_sm100_supported(const AttnArgs& a) { return a.dtype == PG_BF16 && a.d == 128; }

pg_status launch_dq_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse2, const float* Dbuf, void* dq,
                          const float2* rope_tab) {
  const pg_layout* L = a.layout;
  const int64_t T = L->total_tokens;
  CUtensorMap tq, tdo, tk, tv;
  pg_status st = make_tmap_2d_bf16(&tq, q, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 2, 64, BM);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tdo, dO, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 2, 64, BM);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tk, k, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tv, v, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st != PG_OK) return st;
  const size_t smem = sizeof(DqSmem) + 1024;
  st = cuda_check(cudaFuncSetAttribute(attn_dq_sm100_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                  "dq smem attribute");
  if (st != PG_OK) return st;
  prof_begin(PG_KERNEL_BWD_DQ, a.stream);
  attn_dq_sm100_kernel<<<(unsigned)(L->n_tiles[FWD128] * a.Hq), NTHREADS, smem, a.stream>>>(
      tq, tdo, tk, tv, static_cast<__nv_bfloat16*>(dq), lse2, Dbuf, padded_tokens(L), tokens(L),
      tiles<FwdTile>(L, FWD128), intervals(L), a.Hq, a.Hkv, (int)T, a.scale * kLog2e, a.scale,
      rope_tab,
      order_chunk(a.Hq, 1), 2000000000ull);
  prof_end(PG_KERNEL_BWD_DQ, a.stream);
  return cuda_check(cudaGetLastError(), "dq sm100 launch");
}

pg_status read_status_dq_sm100(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_dq, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_dq, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}

}  // namespace pg
