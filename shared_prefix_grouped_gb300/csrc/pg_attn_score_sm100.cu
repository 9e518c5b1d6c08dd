// Responses-only grouped-attention forward on the 5th-generation tensor cores (bf16, head_dim 128):
// scoring many short responses against one long shared context (Pith review of Prefix Grouper,
// "Core claim": the same sharing pattern serves judging many short questions against one long
// context).  Each response row attends to its group's whole prefix and causally to its own
// response; the prefix rows themselves are not queried.
//
// With few query rows per key this is a memory-bound problem: the work per prefix K/V row is
// (response rows) x (query heads per key/value head) dot products, far below the tensor cores'
// FLOP-per-byte ridge.  So the kernel is organised around reading each prefix K/V row once per
// key/value head:
//   * a CTA owns one key/value head kh and up to 256 query rows, which are (token, head) pairs of
//     the Hq / Hkv query heads sharing kh (row m = token (m / hp), head kh * hp + m % hp), loaded
//     by one 3-D TMA box per 64-dim half;
//   * the prefix keys of a group are split into `nsplit` chunks, one per CTA (the grid is
//     spans x row blocks x Hkv x nsplit), so that enough CTAs stream K/V at once to keep HBM busy;
//     split 0 also visits the responses' own keys;
//   * every CTA writes its partial O (fp32, normalised by its own row sum) and its log2-domain LSE;
//     score_combine_kernel merges the splits by their LSEs.  With nsplit == 1 the CTA writes the
//     final bf16 O and natural-log LSE itself.
// Pipeline and warp roles are those of the training forward: 128-key K / V tiles (3-stage K and
// 2-stage V rings, K one tile ahead), S_i = Q_i K^T (M 128 x N 128 x K 128) in TMEM columns
// [128 i, 128 i + 128) with P_i written over its first 64 columns, O_i in [256 + 128 i, ...), one
// MMA-issuing thread (warp 1) whose issue order keeps P_i read before S_i is overwritten, warp 0
// the TMA producer, warps 2..9 the row softmax of query tiles 0 and 1 (one thread per row).  Every
// mbarrier wait is bounded (PG_ERR_TIMEOUT in the status word, then an orderly exit).
#include <math.h>

#include <algorithm>

#include "pg_internal.h"
#include "pg_rowsoftmax.cuh"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;
using namespace rowsoftmax;

namespace {

constexpr int D = 128;
constexpr int BM = 128;                      // rows per query tile (two per CTA)
constexpr int ROWS = 2 * BM;                 // query rows per CTA
constexpr int BN = 128;                      // keys per K/V tile
constexpr int NSK = 3;                       // K pipeline stages
constexpr int NSV = 2;                       // V pipeline stages
constexpr uint32_t QH = ROWS * 128;          // one 64-dim half of the 256 query rows: 32 KiB
constexpr uint32_t KHALF = BN * 64 * 2;      // [128 keys][64 dims] bf16: 16 KiB
constexpr int NTHREADS = 320;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;

__device__ int s_status_score = 0;

struct ScoreSmem {
  uint8_t q[2][QH];            // [dim half][256 rows x 128 bytes]
  uint8_t k[NSK][2 * KHALF];
  uint8_t v[NSV][2 * KHALF];
  uint64_t q_full;
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2];          // S of [query tile] complete
  uint64_t p_full[2];          // P of [query tile] written (its 4 softmax warps)
  uint64_t pv_done[2];         // the P V product of [query tile] has completed
  uint64_t mma_done;
  uint32_t tmem;
};
// The 1024-byte alignment slack included, within the 227 KB a CTA may use.
static_assert(sizeof(ScoreSmem) + 1024 <= 232448, "scoring shared memory");

__device__ __forceinline__ void fail(int code) { atomicCAS(&s_status_score, 0, code); }

// Which CTA does what.  blockIdx.x = ((span * Hkv + kh) * nsplit + c) * nrb + rb, so the row
// blocks that read the same K/V chunk run side by side and share it through L2; the CTA's slot
// within its split is blk = (span * Hkv + kh) * nrb + rb.
struct Work {
  int kh, c, blk;        // key/value head, split, CTA index within the split
  int t0, t_end;         // tokens [t0, t_end) of this row block (all response rows of one group)
  int rows;              // valid query rows = (t_end - t0) * hp
  int p_lo, p_hi;        // prefix keys of this split
  int s_lo, s_hi;        // response keys (split 0 only)
  int n_a, n;            // key tiles: prefix part, total
  int last_tok[2];       // last token of each query tile (-1: tile empty)
  __device__ bool init(const FwdTile* spans, const int4* tok, int Hkv, int hp, int TB, int nrb,
                       int nsplit) {
    int x = blockIdx.x;
    const int rb = x % nrb;
    x /= nrb;
    c = x % nsplit;
    x /= nsplit;
    kh = x % Hkv;
    const int span = x / Hkv;
    blk = (span * Hkv + kh) * nrb + rb;
    const FwdTile sp = spans[span];
    t0 = sp.q0 + rb * TB;
    if (t0 >= sp.q1) return false;
    t_end = min(t0 + TB, sp.q1);
    rows = (t_end - t0) * hp;
    const int lp = sp.p_end - sp.g0;
    const int chunk = ((lp + nsplit - 1) / nsplit + BN - 1) / BN * BN;
    p_lo = min(sp.g0 + c * chunk, sp.p_end);
    p_hi = min(p_lo + chunk, sp.p_end);
    if (c == 0) {
      s_lo = tok[t0].z;          // first row of the first token's own response
      s_hi = t_end;
    } else {
      s_lo = s_hi = 0;
    }
    n_a = (p_hi - p_lo + BN - 1) / BN;
    n = n_a + (s_hi - s_lo + BN - 1) / BN;
    last_tok[0] = t0 + (min(rows, BM) - 1) / hp;
    last_tok[1] = rows > BM ? t_end - 1 : -1;
    return true;
  }
  __device__ void get(int j, int& kt, int& hi) const {
    if (j < n_a) {
      kt = p_lo + j * BN;
      hi = p_hi;
    } else {
      kt = s_lo + (j - n_a) * BN;
      hi = s_hi;
    }
  }
  // Query tile i needs key tile j: every prefix tile; a response tile only up to its last token.
  __device__ bool rel(int i, int j) const {
    if (last_tok[i] < 0) return false;
    if (j < n_a) return true;
    int kt, hi;
    get(j, kt, hi);
    return kt <= last_tok[i];
  }
};

__global__ void __launch_bounds__(NTHREADS, 1)
attn_score_sm100_kernel(const __grid_constant__ CUtensorMap tq,
                        const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, __nv_bfloat16* __restrict__ o,
                        float* __restrict__ lse, float* __restrict__ part_o,
                        float* __restrict__ part_lse, const int4* __restrict__ tok,
                        const FwdTile* __restrict__ spans, int Hq, int Hkv, int hp, int TB,
                        int nrb, int nsplit, int nblk, int Ttot, float scale_log2,
                        uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  ScoreSmem& sm = *reinterpret_cast<ScoreSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Work wk;
  if (!wk.init(spans, tok, Hkv, hp, TB, nrb, nsplit)) return;   // row block past the group's end
  if (wk.t0 < 0 || wk.t_end > Ttot || wk.p_lo < 0 || wk.s_hi > Ttot) {
    if (threadIdx.x == 0) fail(PG_ERR_DEVICE);
    return;
  }
  const bool partial = nsplit > 1;
  const size_t slot = (size_t)wk.c * nblk + wk.blk;
  if (wk.n == 0) {
    // An empty split (the group's prefix is shorter than the others'): contributes nothing.
    if (partial)
      for (int m = threadIdx.x; m < wk.rows; m += NTHREADS) part_lse[slot * ROWS + m] = -INFINITY;
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&sm.q_full, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 4);   // softmax warps of the tile
      mbar_init(&sm.pv_done[i], 1);
    }
    mbar_init(&sm.mma_done, 1);
    fence_mbar_init();
  }
  // Rows past the TMA box (when hp does not divide 256) are zeroed so the MMAs read finite data.
  const int box_rows = TB * hp;
  if (box_rows < ROWS) {
    for (int idx = threadIdx.x; idx < 2 * (ROWS - box_rows) * 8; idx += NTHREADS) {
      const int hf = idx / ((ROWS - box_rows) * 8), rem = idx % ((ROWS - box_rows) * 8);
      *reinterpret_cast<uint4*>(sm.q[hf] + (box_rows + rem / 8) * 128 + (rem % 8) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer -----
    // Q once (one 3-D box per 64-dim half), then K tiles into a 3-stage ring and V tiles into a
    // 2-stage ring, K one tile ahead of V (the score product of a tile precedes its P V product).
    if (elect_one()) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      const int xk = wk.kh * D;
      mbar_expect_tx(&sm.q_full, 2 * box_rows * 128);
      tma_load_3d(sm.q[0], &tq, &sm.q_full, 0, wk.kh * hp, wk.t0);
      tma_load_3d(sm.q[1], &tq, &sm.q_full, 64, wk.kh * hp, wk.t0);
      int k_issued = 0, v_issued = 0;
      auto load_k = [&](int j) -> bool {
        const int s = j % NSK;
        if (!mbar_wait(&sm.k_empty[s], ((j / NSK) & 1) ^ 1, wait_ns)) return false;
        int kt, hi;
        wk.get(j, kt, hi);
        mbar_expect_tx(&sm.k_full[s], 2 * KHALF);
        tma_load_2d(sm.k[s], &tk, &sm.k_full[s], xk, kt);
        tma_load_2d(sm.k[s] + KHALF, &tk, &sm.k_full[s], xk + 64, kt);
        ++k_issued;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % NSV;
        if (!mbar_wait(&sm.v_empty[s], ((j / NSV) & 1) ^ 1, wait_ns)) return false;
        int kt, hi;
        wk.get(j, kt, hi);
        mbar_expect_tx(&sm.v_full[s], 2 * KHALF);
        tma_load_2d(sm.v[s], &tv, &sm.v_full[s], xk, kt);
        tma_load_2d(sm.v[s] + KHALF, &tv, &sm.v_full[s], xk + 64, kt);
        ++v_issued;
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; ok && j < wk.n; ++j) {
        if (j + 1 < wk.n && !load_k(j + 1)) { ok = false; break; }
        if (!load_v(j)) { ok = false; break; }
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      // Leave no copy in flight: the last stages' loads must have landed before exit.
      mbar_wait(&sm.q_full, 0, wait_ns);
      for (int j = (k_issued > NSK ? k_issued - NSK : 0); j < k_issued; ++j)
        mbar_wait(&sm.k_full[j % NSK], (j / NSK) & 1, wait_ns);
      for (int j = (v_issued > NSV ? v_issued - NSV : 0); j < v_issued; ++j)
        mbar_wait(&sm.v_full[j % NSV], (j / NSV) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer -------
    // One thread issues every product, in the order P V of tile 0 (key tile j), S of tile 0
    // (j + 1), P V of tile 1 (j), S of tile 1 (j + 1): the tensor core executes them in issue
    // order, so P_i(j), written over S_i's first 64 columns, is read before S_i(j + 1) lands there.
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      // V as the MN-major B operand of P V: the two 64-dim halves are LBO apart.
      const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), KHALF, 1024);
      int n_pv[2] = {0, 0};
      bool ok = mbar_wait(&sm.q_full, 0, wait_ns);
      auto wait_k = [&](int j) { return mbar_wait(&sm.k_full[j % NSK], (j / NSK) & 1, wait_ns); };
      auto wait_v = [&](int j) { return mbar_wait(&sm.v_full[j % NSV], (j / NSV) & 1, wait_ns); };
      // S_i(j): query tile i (rows [128 i, 128 i + 128) of each Q half) against key tile j.
      auto issue_s = [&](int i, int j) {
        tc_fence_after();
        const uint64_t qd = desc_add(qd0, i * BM * 128);
        const uint64_t kd = desc_add(kd0, (j % NSK) * 2 * KHALF);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + 128 * i, desc_add(qd, (kk >> 2) * QH + (kk & 3) * 32),
                 desc_add(kd, (kk >> 2) * KHALF + (kk & 3) * 32), idesc_s, kk != 0);
        mma_commit(&sm.s_full[i]);
      };
      // O_i += P_i(j) V_j, P_i read from the first 64 columns of S_i.
      auto issue_pv = [&](int i, int j) -> bool {
        if (!mbar_wait(&sm.p_full[i], n_pv[i] & 1, wait_ns)) return false;
        tc_fence_after();
        const uint64_t vd = desc_add(vd0, (j % NSV) * 2 * KHALF);
        const uint32_t acc0 = n_pv[i] != 0;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + 256 + 128 * i, tmem + 128 * i + kk * 8, desc_add(vd, kk * 2048), idesc_pv,
                 kk == 0 ? acc0 : 1u);
        mma_commit(&sm.pv_done[i]);
        ++n_pv[i];
        return true;
      };
      if (ok) {
        ok = wait_k(0);
        for (int i = 0; ok && i < 2; ++i)
          if (wk.rel(i, 0)) issue_s(i, 0);
        mma_commit(&sm.k_empty[0]);
      }
      for (int j = 0; ok && j < wk.n; ++j) {
        const bool more = j + 1 < wk.n;
        if (!wait_v(j)) { ok = false; break; }
        bool k_ready = !more;
        for (int i = 0; ok && i < 2; ++i) {
          if (wk.rel(i, j) && !issue_pv(i, j)) { ok = false; break; }
          if (more && wk.rel(i, j + 1)) {
            if (!k_ready && !(k_ready = wait_k(j + 1))) { ok = false; break; }
            issue_s(i, j + 1);
          }
        }
        if (!ok) break;
        if (!k_ready && !wait_k(j + 1)) { ok = false; break; }
        mma_commit(&sm.v_empty[j % NSV]);
        if (more) mma_commit(&sm.k_empty[(j + 1) % NSK]);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax ----------
    const int i = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int m = i * BM + quarter * 32 + lane;      // query row of the CTA
    const bool active = wk.last_tok[i] >= 0;
    const bool valid = active && m < wk.rows;
    const int t = wk.t0 + (valid ? m / hp : 0);
    const int h = wk.kh * hp + m % hp;
    const int own_lo = tok[t].z;
    const bool any_valid = __any_sync(0xffffffffu, valid);
    // The unmasked path is chosen per warp: its TMEM stores are warp-collective, so every lane of
    // a warp must take the same path (a warp that mixes padding and real rows takes the masked one).
    const bool all_valid = __all_sync(0xffffffffu, valid);
    const bool o_al32 = (reinterpret_cast<uintptr_t>(o) & 31) == 0;
    const bool p_al32 = (reinterpret_cast<uintptr_t>(part_o) & 31) == 0;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + 128 * i + lane_addr, t_o = tmem + 256 + 128 * i + lane_addr;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    int c = 0;
    for (int j = 0; active && j < wk.n; ++j) {
      if (!wk.rel(i, j)) continue;
      int kt, hi;
      wk.get(j, kt, hi);
      if (!warp_wait(&sm.s_full[i], c & 1, wait_ns)) { ok = false; break; }
      if (!any_valid) {
        // Padding rows only (the block has fewer than 256 query rows): keep the barrier protocol
        // and nothing else.  Their S columns go to the P V product as they are, so their O rows
        // hold garbage that is never stored.
        ++c;
        warp_arrive(&sm.p_full[i]);
        continue;
      }
      tc_fence_after();
      // Prefix keys are visible to every response row; response keys from the row's own response
      // start up to the row itself: one contiguous run [lo, lo + len) of the tile's columns
      // (empty for padding rows).  Row handling as in the training forward: 64 columns at a time;
      // an exact pass on the first tile and whenever a row's max grows past the rescale threshold,
      // otherwise one pass straight to P against the running reference.
      const bool prefix = j < wk.n_a;
      const bool full_tile = prefix && all_valid && kt + BN <= hi;
      const int lo = prefix ? 0 : max(own_lo - kt, 0);
      const int len = valid ? max(min(hi, prefix ? hi : t + 1) - kt - lo, 0) : 0;
      uint32_t sr[64];
      bool stored = false;
      if (c > 0) {
        uint32_t pa[32], pb[32];
        float mxk = -INFINITY;
        const float mref0 = (m_used == -INFINITY) ? 0.f : m_used;
        load64(t_s, sr);
        const float sa = full_tile ? exp64_keep<false>(sr, 0, lo, len, scale_log2, mref0, pa, mxk)
                                   : exp64_keep<true>(sr, 0, lo, len, scale_log2, mref0, pa, mxk);
        load64(t_s + 64, sr);
        const float sb = full_tile ? exp64_keep<false>(sr, 64, lo, len, scale_log2, mref0, pb, mxk)
                                   : exp64_keep<true>(sr, 64, lo, len, scale_log2, mref0, pb, mxk);
        const bool grow = fmaxf(m_used, mxk * scale_log2) > m_used + kRescaleThreshold;
        if (!__any_sync(0xffffffffu, grow)) {
          tmem_st16(t_s, pa);
          tmem_st16(t_s + 16, pa + 16);
          tmem_st16(t_s + 32, pb);
          tmem_st16(t_s + 48, pb + 16);
          l += sa;
          l += sb;
          stored = true;
        }
      }
      if (!stored) {
        load64(t_s + 64, sr);
        float mx = full_tile ? max64<false>(sr, 64, lo, len) : max64<true>(sr, 64, lo, len);
        load64(t_s, sr);
        mx = fmaxf(mx, full_tile ? max64<false>(sr, 0, lo, len) : max64<true>(sr, 0, lo, len));
        const float m_new = fmaxf(m_used, mx * scale_log2);
        const bool rescale = m_new > m_used + kRescaleThreshold;   // false when m_new is -inf
        float corr = 1.f;
        if (rescale) {
          corr = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
          m_used = m_new;
          l *= corr;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        // Rescaling O needs the previous key tile's P V product done (its S completed after it).
        const bool any_rescale = __any_sync(0xffffffffu, rescale) && c > 0;
        if (any_rescale) {
          if (!warp_wait(&sm.pv_done[i], (c - 1) & 1, wait_ns)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t orr[32];
            tmem_ld32(t_o + q4 * 32, orr);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * corr);
            tmem_st32(t_o + q4 * 32, orr);
          }
        }
        l += full_tile ? exp64<false>(sr, 0, lo, len, scale_log2, mref, t_s)
                       : exp64<true>(sr, 0, lo, len, scale_log2, mref, t_s);
        load64(t_s + 64, sr);
        l += full_tile ? exp64<false>(sr, 64, lo, len, scale_log2, mref, t_s + 32)
                       : exp64<true>(sr, 64, lo, len, scale_log2, mref, t_s + 32);
      }
      tmem_st_wait();
      ++c;
      tc_fence_before();
      warp_arrive(&sm.p_full[i]);
    }
    // Epilogue: O / l with the LSE, final (one split) or partial (fp32, log2-domain LSE).
    if (active && ok && c > 0 && warp_wait(&sm.pv_done[i], (c - 1) & 1, wait_ns)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const float lse2 = l > 0.f ? m_used + log2f(l) : -INFINITY;
#pragma unroll 1
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t orr[32];
        tmem_ld32(t_o + q4 * 32, orr);
        tmem_ld_wait();
        if (!valid) continue;
        // 32-byte stores where the buffer is 32-byte aligned (rows are 256 or 512 bytes apart).
        if (partial) {
          float* prow = part_o + (slot * ROWS + m) * D + q4 * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = __float_as_uint(__uint_as_float(orr[e + u]) * inv);
            if (p_al32) {
              st_global_v8(prow + e, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            } else {
              *reinterpret_cast<uint4*>(prow + e) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(prow + e + 4) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        } else {
          __nv_bfloat16* orow = o + ((size_t)t * Hq + h) * D + q4 * 32;
#pragma unroll
          for (int e = 0; e < 32; e += 16) {
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              w[u] = pack_bf16x2(__uint_as_float(orr[e + 2 * u]) * inv,
                                 __uint_as_float(orr[e + 2 * u + 1]) * inv);
            if (o_al32) {
              st_global_v8(orow + e, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
            } else {
              *reinterpret_cast<uint4*>(orow + e) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(orow + e + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
      if (valid) {
        if (partial)
          part_lse[slot * ROWS + m] = lse2;
        else
          lse[(size_t)h * Ttot + t] = lse2 * kLn2;
      }
    } else if (active && c > 0) {
      ok = false;
    } else if (valid && partial) {
      part_lse[slot * ROWS + m] = -INFINITY;      // no key tile reached this row in this split
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

// Merge of the splits: four warps per query row of a CTA slot (a block of 256 threads takes two
// rows); warp w of a row accumulates splits w, w + 4, ..., lane l owns dims [4 l, 4 l + 4), and the
// four partial sums meet in shared memory.
// O = sum_c 2^(lse_c - M) O_c / sum_c 2^(lse_c - M), LSE = (M + log2 sum_c 2^(lse_c - M)) ln 2,
// with M the largest split LSE; splits that saw no key (LSE -inf) drop out.  Every warp of a row
// reads all split LSEs (split c by lane c % 32) and forms M and the weights itself.
constexpr int kMergeWarpsPerRow = 4;

__global__ void __launch_bounds__(256)
score_combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                     const FwdTile* __restrict__ spans, int Hq, int Hkv, int hp, int TB, int nrb,
                     int nsplit, int nblk, int Ttot) {
  __shared__ float4 red[2][kMergeWarpsPerRow][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rl = warp / kMergeWarpsPerRow, wr = warp % kMergeWarpsPerRow;   // row in block, part
  const int64_t row = (int64_t)blockIdx.x * 2 + rl;
  bool valid = row < (int64_t)nblk * ROWS;
  int blk = 0, m = 0, t = 0, h = 0;
  if (valid) {
    blk = (int)(row / ROWS);
    m = (int)(row % ROWS);
    const int rb = blk % nrb;
    const int kh = (blk / nrb) % Hkv;
    const FwdTile sp = spans[blk / nrb / Hkv];
    const int t0 = sp.q0 + rb * TB;
    valid = t0 < sp.q1 && m < (min(t0 + TB, sp.q1) - t0) * hp;
    t = t0 + m / hp;
    h = kh * hp + m % hp;
  }
  const size_t stride = (size_t)nblk * ROWS;
  float M = -INFINITY, wa = 0.f, wb = 0.f, W = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (valid) {    // uniform per warp
    // nsplit <= 64: lane l holds the LSEs of splits l and l + 32.
    const float* pl = part_lse + (size_t)blk * ROWS + m;
    const float la = lane < nsplit ? pl[lane * stride] : -INFINITY;
    const float lb = lane + 32 < nsplit ? pl[(lane + 32) * stride] : -INFINITY;
    M = fmaxf(la, lb);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    wa = M == -INFINITY ? 0.f : exp2f(la - M);     // exp2(-inf) = 0 for empty splits
    wb = M == -INFINITY ? 0.f : exp2f(lb - M);
    W = wa + wb;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
    const float* po = part_o + ((size_t)blk * ROWS + m) * D + 4 * lane;
    const size_t ostride = stride * D;
    for (int c0 = wr; c0 < nsplit; c0 += 4 * kMergeWarpsPerRow) {
      float w[4];
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * kMergeWarpsPerRow;
        const int cc = c < nsplit ? c : 0;
        const float wc = __shfl_sync(0xffffffffu, cc < 32 ? wa : wb, cc & 31);
        w[u] = c < nsplit ? wc : 0.f;
        v[u] = w[u] > 0.f ? *reinterpret_cast<const float4*>(po + (size_t)c * ostride)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
      }
    }
  }
  red[rl][wr][lane] = acc;
  __syncthreads();
  if (!valid || wr != 0) return;
#pragma unroll
  for (int i = 1; i < kMergeWarpsPerRow; ++i) {
    const float4 x = red[rl][i][lane];
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  uint2 packed;
  packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(o + ((size_t)t * Hq + h) * D + 4 * lane) = packed;
  if (lane == 0) lse[(size_t)h * Ttot + t] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
}

}  // namespace

bool score_sm100_supported(const AttnArgs& a) {
  return a.dtype == PG_BF16 && a.d == 128 && a.Hq / a.Hkv <= ROWS;
}

ScorePlan score_plan(const pg_layout* L, int Hq, int Hkv) {
  ScorePlan p{};
  p.hp = Hq / Hkv;
  p.TB = ROWS / p.hp;
  p.nrb = (int)std::max<int64_t>(1, (L->max_response_rows + p.TB - 1) / p.TB);
  p.nblk = L->n_tiles[SPANS] * p.nrb * Hkv;
  // As many splits as fit in one wave of the 152 SMs, each split keeping at least two key tiles.
  constexpr int64_t kTargetCtas = 152;
  int64_t ns = p.nblk == 0 ? 1 : std::max<int64_t>(1, kTargetCtas / p.nblk);
  ns = std::min<int64_t>(ns, 64);
  ns = std::min<int64_t>(ns, std::max<int64_t>(1, L->max_position / (2 * BN)));
  p.nsplit = (int)ns;
  if (p.nsplit > 1) {
    p.part_o_bytes = (size_t)p.nsplit * p.nblk * ROWS * D * sizeof(float);
    p.part_lse_bytes = (size_t)p.nsplit * p.nblk * ROWS * sizeof(float);
  }
  return p;
}

pg_status launch_score_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                             void* o, float* lse, float* part_o, float* part_lse) {
  const pg_layout* L = a.layout;
  const int64_t T = L->total_tokens;
  const ScorePlan p = score_plan(L, a.Hq, a.Hkv);
  if (p.nblk == 0) return PG_OK;                 // no response rows at all
  CUtensorMap tq, tk, tv;
  pg_status st = make_tmap_3d_bf16(&tq, q, D, (uint64_t)a.Hq, (uint64_t)T, D * 2,
                                   (uint64_t)a.Hq * D * 2, 64, (uint32_t)p.hp, (uint32_t)p.TB);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tk, k, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st == PG_OK)
    st = make_tmap_2d_bf16(&tv, v, (uint64_t)a.Hkv * D, T, (uint64_t)a.Hkv * D * 2, 64, BN);
  if (st != PG_OK) return st;
  const size_t smem = sizeof(ScoreSmem) + 1024;
  st = cuda_check(cudaFuncSetAttribute(attn_score_sm100_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem),
                  "score smem attribute");
  if (st != PG_OK) return st;
  const uint64_t wait_ns = 2000000000ull;
  prof_begin(PG_KERNEL_ATTN_FWD, a.stream);
  attn_score_sm100_kernel<<<(unsigned)(p.nblk * p.nsplit), NTHREADS, smem, a.stream>>>(
      tq, tk, tv, static_cast<__nv_bfloat16*>(o), lse, part_o, part_lse, tokens(L),
      tiles<FwdTile>(L, SPANS), a.Hq, a.Hkv, p.hp, p.TB, p.nrb, p.nsplit, (int)p.nblk, (int)T,
      a.scale * kLog2e, wait_ns);
  prof_end(PG_KERNEL_ATTN_FWD, a.stream);
  st = cuda_check(cudaGetLastError(), "score sm100 launch");
  if (st != PG_OK || p.nsplit == 1) return st;
  const int64_t rows = p.nblk * ROWS;
  prof_begin(PG_KERNEL_SCORE_COMBINE, a.stream);
  score_combine_kernel<<<(unsigned)((rows + 1) / 2), 256, 0, a.stream>>>(
      part_o, part_lse, static_cast<__nv_bfloat16*>(o), lse, tiles<FwdTile>(L, SPANS), a.Hq,
      a.Hkv, p.hp, p.TB, p.nrb, p.nsplit, (int)p.nblk, (int)T);
  prof_end(PG_KERNEL_SCORE_COMBINE, a.stream);
  return cuda_check(cudaGetLastError(), "score combine launch");
}

pg_status read_status_score_sm100(bool clear, int32_t* code) {
  int32_t v = 0;
  pg_status st = cuda_check(cudaMemcpyFromSymbol(&v, s_status_score, sizeof(v)), "read status");
  if (st != PG_OK) return st;
  if (clear && v != 0) {
    int32_t z = 0;
    st = cuda_check(cudaMemcpyToSymbol(s_status_score, &z, sizeof(z)), "clear status");
    if (st != PG_OK) return st;
  }
  if (*code == 0) *code = v;
  return PG_OK;
}

}  // namespace pg
