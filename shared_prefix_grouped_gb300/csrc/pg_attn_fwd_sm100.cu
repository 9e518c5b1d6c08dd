// Grouped-attention forward on the 5th-generation tensor cores (bf16, head_dim 128).
//
// One CTA owns up to 256 packed query rows of one group -- two 128-row query tiles -- and one
// query head (a 256-row FwdTile), and streams the key/value tiles those rows can see: the group's
// prefix [g0, p_end) -- every response row sees all of it, prefix rows causally -- then the
// responses' part [s_lo, s_hi) (Pith review of Prefix Grouper, "What carries the argument": prefix
// self-attention plus suffix attention over the prefix and the row's own response).  Both query
// tiles share each K/V tile loaded into shared memory, and all CTAs of a group read the same
// prefix K/V tiles, which stay resident in L2 across the group's query tiles and heads.
//
// Warp roles (352 threads):
//   warp 0      TMA producer: Q tiles once, then 64-key K and V tiles into a 4-stage ring
//   warp 1      TMEM allocation and the score MMAs, warp 10 the P V MMAs (one elected thread
//               each, so both kinds are queued on the tensor core at once), per key tile j and
//               query tile i:
//                 S_i = Q_i K_j^T   (M 128 x N 64 keys x K 128; fp32 TMEM columns [64 i, 64 i + 64))
//                 O_i += P_i V_j    (M 128 x N 128 dims x K 64; fp32 TMEM columns [128 + 128 i, ...)),
//                                   with P_i read from TMEM (bf16, columns [384 + 64 i + 32 b, ...)
//                                   for buffer b) and V from shared memory
//   warps 2..5  softmax of query tile 0, warps 6..9 of query tile 1: one thread per query row
//               (TMEM lane = row); S from TMEM to registers, masking, online max / sum in fp32
//               (exp2 with the scale folded in), P rounded to bf16 and stored into TMEM (the A
//               operand of P V, double-buffered), O rescaled in TMEM only when the running max
//               grows by more than 2^8, and the final O / l, LSE epilogue.
// A key tile that lies entirely after the last row of query tile 0 is skipped for that tile.
//
// Every mbarrier wait is bounded (PG_ERR_TIMEOUT in the status word, then an orderly exit: copies
// in flight are awaited, MMAs committed, TMEM freed).
#include <math.h>

#include "pg_internal.h"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;

namespace {

constexpr int D = 128;          // head_dim
constexpr int BM = 128;         // query rows per query tile (two per CTA)
constexpr int BN = 64;          // keys per tile
constexpr int NS = 4;           // K/V pipeline stages
constexpr uint32_t QHALF = BM * 64 * 2;    // [128 rows][64 dims] bf16: 16 KiB
constexpr uint32_t KHALF = BN * 64 * 2;    // [64 keys][64 dims] bf16: 8 KiB
constexpr int NTHREADS = 352;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ int s_status_fwd = 0;

// Key tile j of a CTA: the tiles of its causal key ranges (the group's prefix, or a nested
// prefix's ancestors) first, then of its own range; and which query tiles need it.  Built once per
// CTA in shared memory.
struct Plan {
  int n_r, n_a, n;                  // key ranges, key tiles in causal ranges, all key tiles
  int lo[kMaxKeyRanges], hi[kMaxKeyRanges], cum[kMaxKeyRanges + 1];
  int q0, q1;
  int last[2];      // last query row of each query tile (-1: tile empty)
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
    q0 = t.q0;
    q1 = t.q1;
    last[0] = min(q0 + BM, q1) - 1;
    last[1] = (q1 > q0 + BM) ? q1 - 1 : -1;
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

struct FwdSmem {
  uint8_t q[2][2 * QHALF];
  uint8_t k[NS][2 * KHALF];
  uint8_t v[NS][2 * KHALF];
  uint64_t q_full;
  uint64_t k_full[NS], v_full[NS], kv_empty[NS];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2][2];    // P of [query tile][buffer] written
  uint64_t pv_done[2][2];   // the P V product reading [query tile][buffer] has completed
  uint64_t mma_done, mma_done2;
  uint32_t tmem;
  Plan plan;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fail(int code) { atomicCAS(&s_status_fwd, 0, code); }

__global__ void __launch_bounds__(NTHREADS, 1)
attn_fwd_sm100_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, const int4* __restrict__ tok,
                      const FwdTile* __restrict__ tiles, const int2* __restrict__ ivs,
                      float* __restrict__ lse2_out, int64_t ldl, int Hq, int Hkv, int Ttot,
                      float scale_log2, uint64_t wait_ns, uint32_t debug) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile_id = blockIdx.x / Hq, h = blockIdx.x % Hq;
  const int kh = h / (Hq / Hkv);
  const FwdTile tl = tiles[tile_id];
  if (tl.q0 < 0 || tl.q1 > Ttot || tl.q0 >= tl.q1 || tl.q1 - tl.q0 > 2 * BM || tl.g0 < 0 ||
      tl.s_hi > Ttot || tl.a_cnt < 0 || tl.a_cnt > kMaxExtraRanges) {
    if (threadIdx.x == 0) fail(PG_ERR_DEVICE);
    return;
  }
  const int nq = (tl.q1 > tl.q0 + BM) ? 2 : 1;

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.s_free[i], 128);
      for (int b = 0; b < 2; ++b) {
        mbar_init(&sm.p_full[i][b], 128);
        mbar_init(&sm.pv_done[i][b], 1);
      }
    }
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
  const Plan& pl = sm.plan;
  const int n = pl.n, n_a = pl.n_a;
  const int last0 = pl.last[0], last1 = pl.last[1];
  // Query tile i needs key tile j unless the tile starts after the query tile's last row.
  auto rel = [&](int i, int kt) { const int l = i ? last1 : last0; return l >= 0 && kt <= l; };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer -----
    if (elect_one()) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      const int xq = h * D, xk = kh * D;
      mbar_expect_tx(&sm.q_full, nq * 2 * QHALF);
      for (int i = 0; i < nq; ++i) {
        tma_load_2d(sm.q[i], &tq, &sm.q_full, xq, tl.q0 + i * BM);
        tma_load_2d(sm.q[i] + QHALF, &tq, &sm.q_full, xq + 64, tl.q0 + i * BM);
      }
      int issued = 0;
      TileCursor cur(pl);
      for (int j = 0; j < n; ++j) {
        const int s = j % NS;
        if (!mbar_wait(&sm.kv_empty[s], ((j / NS) & 1) ^ 1, wait_ns)) {
          fail(PG_ERR_TIMEOUT);
          break;
        }
        const int kt = cur.seek(pl, j);
        mbar_expect_tx(&sm.k_full[s], 2 * KHALF);
        tma_load_2d(sm.k[s], &tk, &sm.k_full[s], xk, kt);
        tma_load_2d(sm.k[s] + KHALF, &tk, &sm.k_full[s], xk + 64, kt);
        mbar_expect_tx(&sm.v_full[s], 2 * KHALF);
        tma_load_2d(sm.v[s], &tv, &sm.v_full[s], xk, kt);
        tma_load_2d(sm.v[s] + KHALF, &tv, &sm.v_full[s], xk + 64, kt);
        ++issued;
      }
      // Leave no copy in flight: the last stages' loads must have landed before exit.
      mbar_wait(&sm.q_full, 0, wait_ns);
      for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j) {
        mbar_wait(&sm.k_full[j % NS], (j / NS) & 1, wait_ns);
        mbar_wait(&sm.v_full[j % NS], (j / NS) & 1, wait_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ score MMAs -------
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      int n_s[2] = {0, 0};        // S products issued per query tile
      bool ok = mbar_wait(&sm.q_full, 0, wait_ns);
      // Descriptor bases: buffers of a kind are contiguous, so buffer n is base + n * stride.
      const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      // S_i(j): scores of query tile i against key tile j.  Needs the K tile and the softmax of
      // tile i to have read its previous scores out of TMEM (S_i is single-buffered).
      TileCursor cur(pl);
      for (int j = 0; ok && j < n; ++j) {
        const int kt = cur.seek(pl, j);
        for (int i = 0; i < nq; ++i) {
          if (!rel(i, kt)) continue;
          if (!mbar_wait(&sm.k_full[j % NS], (j / NS) & 1, wait_ns)) { ok = false; break; }
          if (n_s[i] > 0 && !mbar_wait(&sm.s_free[i], (n_s[i] - 1) & 1, wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t qd = desc_add(qd0, i * 2 * QHALF);
          const uint64_t kd = desc_add(kd0, (j % NS) * 2 * KHALF);
          const uint32_t ts = tmem + 64 * i;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss(ts, desc_add(qd, (kk >> 2) * QHALF + (kk & 3) * 32),
                   desc_add(kd, (kk >> 2) * KHALF + (kk & 3) * 32), idesc_s, kk != 0);
          }
          mma_commit(&sm.s_full[i]);
          ++n_s[i];
        }
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      // Every MMA issued above completes before TMEM is released.
      mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, wait_ns);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------------ P V MMAs ---------
    // A second issuing thread: the products of P with V are queued while the next scores are
    // still being issued.  Ordering with the score MMAs goes through the barriers (a key tile's
    // scores completed before its P was written).
    if (elect_one()) {
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      int n_pv[2] = {0, 0};       // P V products issued per query tile
      const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), KHALF, 1024);
      bool ok = true;
      TileCursor cur(pl);
      for (int j = 0; ok && j < n; ++j) {
        const int kt = cur.seek(pl, j);
        if (!mbar_wait(&sm.v_full[j % NS], (j / NS) & 1, wait_ns)) { ok = false; break; }
        for (int i = 0; i < nq && ok; ++i) {
          if (!rel(i, kt)) continue;
          const int b = n_pv[i] & 1;
          if (!mbar_wait(&sm.p_full[i][b], (n_pv[i] >> 1) & 1, wait_ns)) { ok = false; break; }
          tc_fence_after();
          const uint32_t pt = tmem + 384 + 64 * i + 32 * b, to = tmem + 128 + 128 * i;
          const uint64_t vd = desc_add(vd0, (j % NS) * 2 * KHALF);
          const uint32_t acc0 = n_pv[i] != 0;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(to, pt + kk * 8, desc_add(vd, kk * 2048), idesc_pv, kk == 0 ? acc0 : 1u);
          mma_commit(&sm.pv_done[i][b]);
          ++n_pv[i];
        }
        mma_commit(&sm.kv_empty[j % NS]);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.mma_done2);
      mbar_wait(&sm.mma_done2, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax ----------
    const int i = (warp - 2) >> 2;                // query tile of this warpgroup
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;            // query row within the tile
    const int row = tl.q0 + i * BM + r;
    const int qlast = i ? last1 : last0;
    const bool active = qlast >= 0;
    const bool valid = active && row <= qlast;
    const int rowc = valid ? row : (active ? qlast : tl.q0);
    const int4 ti = tok[rowc];                    // {g0, pe, own_lo, pos}
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + 64 * i, t_o = tmem + 128 + 128 * i;
    const int first_row = tl.q0 + i * BM;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int c = 0;
    TileCursor cur(pl);
    for (int j = 0; active && j < n; ++j) {
      const int kt = cur.seek(pl, j);
      const int hi = cur.hi;
      if (!rel(i, kt)) continue;
      if (!warp_wait(&sm.s_full[i], c & 1, wait_ns)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[64];
      tmem_ld32(t_s + lane_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(t_s + lane_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.s_free[i]);
      // Scores in log2 units; mask where the tile is not entirely visible to every row.
      const bool full_tile = (j < n_a) && (kt + BN <= hi) && (kt + BN - 1 <= first_row);
      float mx = -INFINITY;
      if (full_tile) {
#pragma unroll
        for (int cc = 0; cc < BN; ++cc) {
          const float x = __uint_as_float(sr[cc]) * scale_log2;
          sr[cc] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      } else {
        // Within one key tile a row's visible keys are one contiguous run of columns: in the
        // prefix range [kt, min(hi, row + 1)); in the responses' range the same run starting no
        // earlier than the row's own response (prefix rows get an empty run there).  One unsigned
        // compare per column, no branches.
        const int lo = (j < n_a) ? 0 : max(ti.z - kt, 0);
        const int len = max(min(hi, rowc + 1) - kt - lo, 0);
#pragma unroll
        for (int cc = 0; cc < BN; ++cc) {
          const bool vis = (unsigned)(cc - lo) < (unsigned)len;
          const float x = vis ? __uint_as_float(sr[cc]) * scale_log2 : -INFINITY;
          sr[cc] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      const float m_new = fmaxf(m_used, mx);
      const bool rescale = m_new > m_used + kRescaleThreshold;   // false when m_new is -inf
      float corr = 1.f;
      if (rescale) {
        corr = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - m_new);
        m_used = m_new;
        l *= corr;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      // P = exp2(s - m), rounded to bf16.
      uint32_t pw[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float p0 = fast_exp2(__uint_as_float(sr[2 * e]) - mref);
        const float p1 = fast_exp2(__uint_as_float(sr[2 * e + 1]) - mref);
        l += p0 + p1;
        pw[e] = pack_bf16x2(p0, p1);
      }
      // P is double-buffered in TMEM: the product that read this buffer two key tiles ago must
      // be done.
      // Rescaling O needs the previous key tile's product done too.
      const int b = c & 1;
      const bool any_rescale = __any_sync(0xffffffffu, rescale) && c > 0;
      if (any_rescale) {
        if (!warp_wait(&sm.pv_done[i][(c - 1) & 1], ((c - 1) >> 1) & 1, wait_ns)) {
          ok = false;
          break;
        }
      }
      if (c >= 2 && !warp_wait(&sm.pv_done[i][b], ((c >> 1) - 1) & 1, wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (any_rescale) {
        tc_fence_after();
        {
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t orr[32];
            tmem_ld32(t_o + lane_addr + q4 * 32, orr);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * corr);
            tmem_st32(t_o + lane_addr + q4 * 32, orr);
          }
          tmem_st_wait();
        }
      }
      tmem_st32(tmem + 384 + 64 * i + 32 * b + lane_addr, pw);
      tmem_st_wait();
      ++c;
      if (debug & PG_DEBUG_WITHHOLD_P) continue;   // test hook: never signal P (bounded waits)
      tc_fence_before();
      mbar_arrive(&sm.p_full[i][b]);
    }
    // Epilogue: O / l and the natural-log LSE.
    if (active && ok && c > 0 &&
        warp_wait(&sm.pv_done[i][(c - 1) & 1], ((c - 1) >> 1) & 1, wait_ns)) {
      tc_fence_after();
      const float inv = 1.f / l;
      __nv_bfloat16* orow = o + ((size_t)rowc * Hq + h) * D;
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t orr[32];
        tmem_ld32(t_o + lane_addr + q4 * 32, orr);
        tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(orr[e]) * inv, __uint_as_float(orr[e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(orr[e + 2]) * inv, __uint_as_float(orr[e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(orr[e + 4]) * inv, __uint_as_float(orr[e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(orr[e + 6]) * inv, __uint_as_float(orr[e + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + q4 * 32 + e) = w;
          }
        }
      }
      if (valid) {
        const float lse_row = (m_used + log2f(l)) * kLn2;
        lse[(size_t)h * Ttot + row] = lse_row;
        // the backward's log2-domain copy, rounded exactly as the preprocess would
        if (lse2_out) lse2_out[(size_t)h * ldl + row] = lse_row * kLog2e;
      }
    } else if (active && c > 0) {
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

bool fwd_sm100_supported(const AttnArgs& a) { return a.dtype == PG_BF16 && a.d == 128; }

pg_status launch_fwd_sm100(const AttnArgs& a, const void* q, const void* k, const void* v, void* o,
                           float* lse, float* lse2_out) {
  const pg_layout* L = a.layout;
  const int64_t T = L->total_tokens;
  CUtensorMap tq, tk, tv;
  pg_status st = make_tmap_2d_bf16(&tq, q, (uint64_t)a.Hq * D, T, (uint64_t)a.Hq * D * 2, 64, BM);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tk, k, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tv, v, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st != PG_OK) return st;
  const size_t smem = sizeof(FwdSmem) + 1024;
  st = cuda_check(cudaFuncSetAttribute(attn_fwd_sm100_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                  "fwd smem attribute");
  if (st != PG_OK) return st;
  const uint64_t wait_ns = (a.debug & PG_DEBUG_WITHHOLD_P) ? 50000000ull : 2000000000ull;
  prof_begin(PG_KERNEL_ATTN_FWD, a.stream);
  attn_fwd_sm100_kernel<<<(unsigned)(L->n_tiles[FWD256] * a.Hq), NTHREADS, smem, a.stream>>>(
      tq, tk, tv, static_cast<__nv_bfloat16*>(o), lse, tokens(L), tiles<FwdTile>(L, FWD256),
      intervals(L), lse2_out, padded_tokens(L), a.Hq, a.Hkv, (int)T, a.scale * kLog2e, wait_ns, a.debug);
  prof_end(PG_KERNEL_ATTN_FWD, a.stream);
  return cuda_check(cudaGetLastError(), "fwd sm100 launch");
}

pg_status read_status_fwd_sm100(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_fwd, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_fwd, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}

}  // namespace pg
