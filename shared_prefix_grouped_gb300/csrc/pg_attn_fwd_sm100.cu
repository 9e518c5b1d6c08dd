// Grouped-attention forward on the 5th-generation tensor cores (bf16, head_dim 128).
//
// A work item is up to 256 packed query rows of one group -- two 128-row query tiles -- and one
// query head (a 256-row FwdTile); its CTA streams the key/value tiles those rows can see: the group's
// prefix [g0, p_end) -- every response row sees all of it, prefix rows causally -- then the
// responses' part [s_lo, s_hi) (Pith review of Prefix Grouper, "What carries the argument": prefix
// self-attention plus suffix attention over the prefix and the row's own response).  Both query
// tiles share each K/V tile loaded into shared memory, and the items run in chunks of query heads
// that share a few key/value heads (the query heads of one KV head side by side on the same query
// tile), so a group's prefix K/V tiles are read from DRAM about once per chunk and served from L2
// to every query tile of the group -- the prefix is encoded once, not once per response.
//
// Key tiles are 128 keys wide, so the score product runs at the full MMA rate (N = 128):
//   S_i = Q_i K_j^T   M 128 rows x N 128 keys x K 128 dims, fp32 in TMEM columns [128 i, 128 i + 128)
//   O_i += P_i V_j    M 128 rows x N 128 dims x K 128 keys, fp32 in TMEM columns [256 + 128 i, ...)
// P_i (bf16) is written over the first 64 columns of S_i, from which the P V product reads it as
// its A operand.  One thread issues every MMA, in the order
//   ... P V of tile 0 (key tile j), S of tile 0 (key tile j + 1), P V of tile 1 (j), S of tile 1 (j + 1) ...
// so the tensor core, which executes a CTA's MMAs in issue order, finishes reading P_i(j) before
// S_i(j + 1) overwrites those columns, and while the softmax of one query tile runs the tensor
// core works on the other tile's products.
//
// The grid has one CTA per work item, but a CTA that has issued every load of its item claims the
// next CTA that has not launched yet (cluster launch control: the hardware cancels that CTA and
// hands over its index) and runs that item too, so each SM keeps one CTA that works through items
// in the hardware's launch order.  Between items nothing drains: the next item's Q tile i loads
// once the current item's last score product of tile i has completed, its K / V tiles follow
// through the same rings, and its first products are issued while the current item's last P V
// products and epilogues run.  The producer publishes each item (tile, head, key-tile plan) in
// one of two shared-memory slots, which the other roles release when they are done with it.
//
// Warp roles (320 threads):
//   warp 0      TMA producer: each item's Q tiles, then 128-key K tiles into a 3-stage ring and V
//               tiles into a 2-stage ring, K one tile ahead of V (K is needed first); claims items
//   warp 1      TMEM allocation and the MMA issuer (one elected thread)
//   warps 2..5  softmax of query tile 0, warps 6..9 of query tile 1: one thread per query row
//               (TMEM lane = row); S from TMEM to registers, masking, online max / sum in fp32
//               (exp2 with the scale folded in), P rounded to bf16 and stored into TMEM, O
//               rescaled in TMEM only when the running max grows by more than 2^8, and the final
//               O / l, LSE epilogue.
// A key tile that lies entirely after the last row of query tile 0 is skipped for that tile.
//
// Every mbarrier wait is bounded (PG_ERR_TIMEOUT in the status word, then an orderly exit: copies
// in flight are awaited, MMAs committed, TMEM freed).
#include <math.h>

#include "pg_internal.h"
#include "pg_rowsoftmax.cuh"
#include "pg_sm100.cuh"
#include "pg_tmap.h"

namespace pg {

using namespace sm100;
using namespace rowsoftmax;

namespace {

constexpr int D = 128;          // head_dim
constexpr int BM = 128;         // query rows per query tile (two per item)
constexpr int BN = 128;         // keys per tile
constexpr int NSK = 3;          // K pipeline stages
constexpr int NSV = 2;          // V pipeline stages
constexpr uint32_t QHALF = BM * 64 * 2;    // [128 rows][64 dims] bf16: 16 KiB
constexpr uint32_t KHALF = BN * 64 * 2;    // [128 keys][64 dims] bf16: 16 KiB
constexpr int NTHREADS = 320;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ int s_status_fwd = 0;

// Key tile j of an item: the tiles of its causal key ranges (the group's prefix, or a nested
// prefix's ancestors) first, then of its own range; and which query tiles need it.  Built by the
// producer in the item's shared-memory slot.
struct Plan {
  int n_r, n_a, n;                  // key ranges, key tiles in causal ranges, all key tiles
  int lo[kMaxKeyRanges], hi[kMaxKeyRanges], cum[kMaxKeyRanges + 1];
  int q0, q1;
  int last[2];      // last query row of each query tile (-1: tile empty)
  int lastj[2];     // last key tile each query tile uses (-1: none)
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
    // Query tile i uses key tile j (first key kt) iff last[i] >= 0 and kt <= last[i].
    for (int i = 0; i < 2; ++i) {
      lastj[i] = -1;
      for (int r = 0; last[i] >= 0 && r < n_r; ++r)
        if (hi[r] > lo[r] && lo[r] <= last[i])
          lastj[i] = max(lastj[i], cum[r] + min(cum[r + 1] - cum[r] - 1, (last[i] - lo[r]) / BN));
    }
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

// A work item as the producer publishes it to the other roles (two slots, alternating).
struct Item {
  int x;                    // item index (a blockIdx.x of the grid); -1: no more work
  int h;                    // query head
  FwdTile tl;
  Plan plan;
};

struct FwdSmem {
  uint8_t q[2][2 * QHALF];
  uint8_t k[NSK][2 * KHALF];
  uint8_t v[NSV][2 * KHALF];
  uint64_t q_full[2], q_empty[2];   // Q of [query tile] loaded / no longer read (once per item)
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2];       // S of [query tile] complete
  uint64_t p_full[2];       // P of [query tile] written (its 4 softmax warps)
  uint64_t pv_done[2];      // the P V product of [query tile] has completed
  uint64_t item_full[2];    // item slot published (producer)
  uint64_t item_empty[2];   // item slot released (the MMA issuer and the 8 softmax warps)
  uint64_t clc_full;        // cluster-launch-control response arrived
  uint64_t mma_done;
  alignas(16) uint4 clc_resp;
  uint32_t tmem;
  Item item[2];
};
// The 1024-byte alignment slack included, within the 227 KB a CTA may use.
static_assert(sizeof(FwdSmem) + 1024 <= 232448, "forward shared memory");

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
                      float scale_log2, int hc, uint64_t wait_ns, uint32_t debug) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>(base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sm.q_full[i], 1);
      mbar_init(&sm.q_empty[i], 1);
      mbar_init(&sm.s_full[i], 1);
      mbar_init(&sm.p_full[i], 4);   // softmax warps of the tile
      mbar_init(&sm.pv_done[i], 1);
      mbar_init(&sm.item_full[i], 1);
      mbar_init(&sm.item_empty[i], 9);   // the MMA issuer and the 8 softmax warps
    }
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&sm.k_full[s], 1);
      mbar_init(&sm.k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&sm.v_full[s], 1);
      mbar_init(&sm.v_empty[s], 1);
    }
    mbar_init(&sm.clc_full, 1);
    mbar_init(&sm.mma_done, 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer -----
    // Publishes each work item (tile, head, key-tile plan) into a slot, loads its Q tiles once
    // the previous item's score products are done with the buffers, streams its K / V tiles
    // through the rings (positions continue across items), then claims the next item.
    if (elect_one()) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      const int n_tiles = gridDim.x / Hq;
      int x = blockIdx.x;
      int k_issued = 0, v_issued = 0, q_loaded[2] = {0, 0};
      uint32_t clc_phase = 0;
      bool ok = true, clc_pending = false;
      for (uint32_t kq = 0;; ++kq) {
        const int slot = kq & 1;
        // The slot's previous item (kq - 2) must be released by every consumer.
        if (kq >= 2 && !mbar_wait(&sm.item_empty[slot], ((kq >> 1) - 1) & 1, wait_ns)) {
          ok = false;
          break;
        }
        Item& it = sm.item[slot];
        if (x >= 0) {
          int tile_id, h;
          chunked_order(x, n_tiles, Hq, hc, tile_id, h);
          const FwdTile tl = tiles[tile_id];
          if (tl.q0 < 0 || tl.q1 > Ttot || tl.q0 >= tl.q1 || tl.q1 - tl.q0 > 2 * BM ||
              tl.g0 < 0 || tl.s_hi > Ttot || tl.a_cnt < 0 || tl.a_cnt > kMaxExtraRanges) {
            fail(PG_ERR_DEVICE);
            x = -1;
          } else {
            it.tl = tl;
            it.h = h;
            it.plan.init(tl, ivs);
          }
        }
        it.x = x;
        mbar_arrive(&sm.item_full[slot]);
        if (x < 0) break;
        const Plan& pl = it.plan;
        const int xq = it.h * D, xk = (it.h / (Hq / Hkv)) * D;
        // Both query tiles' rows are loaded (rows past the tile are read but never used).  They
        // are brought into L2 first: the loads below wait for the previous item's last score
        // products, and from L2 they then land sooner than from DRAM.
        for (int i = 0; kq >= 1 && i < 4; ++i)
          if (it.tl.q0 + (i >> 1) * BM < Ttot)
            tma_prefetch_l2_2d(&tq, xq + (i & 1) * 64, it.tl.q0 + (i >> 1) * BM);
        for (int i = 0; ok && i < 2; ++i) {
          if (kq >= 1 && !mbar_wait(&sm.q_empty[i], (kq - 1) & 1, wait_ns)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&sm.q_full[i], 2 * QHALF);
          tma_load_2d(sm.q[i], &tq, &sm.q_full[i], xq, it.tl.q0 + i * BM);
          tma_load_2d(sm.q[i] + QHALF, &tq, &sm.q_full[i], xq + 64, it.tl.q0 + i * BM);
          ++q_loaded[i];
        }
        if (!ok) break;
        // K(j + 1) is issued before V(j): the score product of key tile j + 1 follows the P V
        // product of key tile j closely, and the deeper K ring gives its load the longer lead.
        const int n = pl.n;
        TileCursor cur(pl);
        auto load_k = [&](int j) -> bool {
          const int p = k_issued, s = p % NSK;
          if (!mbar_wait(&sm.k_empty[s], ((p / NSK) & 1) ^ 1, wait_ns)) return false;
          const int kt = cur.seek(pl, j);
          mbar_expect_tx(&sm.k_full[s], 2 * KHALF);
          tma_load_2d(sm.k[s], &tk, &sm.k_full[s], xk, kt);
          tma_load_2d(sm.k[s] + KHALF, &tk, &sm.k_full[s], xk + 64, kt);
          ++k_issued;
          return true;
        };
        TileCursor vcur(pl);
        auto load_v = [&](int j) -> bool {
          const int p = v_issued, s = p % NSV;
          if (!mbar_wait(&sm.v_empty[s], ((p / NSV) & 1) ^ 1, wait_ns)) return false;
          const int kt = vcur.seek(pl, j);
          mbar_expect_tx(&sm.v_full[s], 2 * KHALF);
          tma_load_2d(sm.v[s], &tv, &sm.v_full[s], xk, kt);
          tma_load_2d(sm.v[s] + KHALF, &tv, &sm.v_full[s], xk + 64, kt);
          ++v_issued;
          return true;
        };
        if (n > 0) ok = load_k(0);
        for (int j = 0; ok && j < n; ++j) {
          if (j + 1 < n && !load_k(j + 1)) { ok = false; break; }
          if (!load_v(j)) { ok = false; break; }
        }
        if (!ok) break;
        // Every load of this item is issued: claim the next item while its tail runs.
        x = clc_claim(&sm.clc_resp, &sm.clc_full, clc_phase, wait_ns);
        if (x == -2) {
          clc_pending = true;
          ok = false;
          break;
        }
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      // Leave nothing in flight: the last loads must have landed, a claim must have answered.
      if (clc_pending) mbar_wait(&sm.clc_full, clc_phase, wait_ns);
      for (int i = 0; i < 2; ++i)
        if (q_loaded[i] > 0) mbar_wait(&sm.q_full[i], (q_loaded[i] - 1) & 1, wait_ns);
      for (int p = (k_issued > NSK ? k_issued - NSK : 0); p < k_issued; ++p)
        mbar_wait(&sm.k_full[p % NSK], (p / NSK) & 1, wait_ns);
      for (int p = (v_issued > NSV ? v_issued - NSV : 0); p < v_issued; ++p)
        mbar_wait(&sm.v_full[p % NSV], (p / NSV) & 1, wait_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer -------
    if (elect_one()) {
      constexpr uint32_t idesc_s = idesc_bf16(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16(BM, D, 0, 1);
      // Descriptor bases: buffers of a kind are contiguous, so buffer n is base + n * stride.
      const uint64_t qd0 = sdesc_sw128(smem_u32(sm.q[0]), 16, 1024);
      const uint64_t kd0 = sdesc_sw128(smem_u32(sm.k[0]), 16, 1024);
      // V as the MN-major B operand of P V: the two 64-dim halves are LBO apart.
      const uint64_t vd0 = sdesc_sw128(smem_u32(sm.v[0]), KHALF, 1024);
      int kbase = 0;              // ring position of the current item's first key tile
      int n_pv[2] = {0, 0};       // P V products issued per query tile, over all items
      bool ok = true;
      for (uint32_t kq = 0; ok; ++kq) {
        const int slot = kq & 1;
        if (!mbar_wait(&sm.item_full[slot], (kq >> 1) & 1, wait_ns)) { ok = false; break; }
        const Item& it = sm.item[slot];
        if (it.x < 0) break;
        const Plan& pl = it.plan;
        const int n = pl.n, last0 = pl.last[0], last1 = pl.last[1];
        const int lastj0 = pl.lastj[0], lastj1 = pl.lastj[1];
        auto rel = [&](int i, int kt) { const int l = i ? last1 : last0; return l >= 0 && kt <= l; };
        if (!mbar_wait(&sm.q_full[0], kq & 1, wait_ns) || !mbar_wait(&sm.q_full[1], kq & 1, wait_ns)) {
          ok = false;
          break;
        }
        // Q_i is released after the item's last score product of query tile i (at once if the
        // tile uses no key tile), so the next item's load overlaps this item's tail.
        if (lastj0 < 0) mma_commit(&sm.q_empty[0]);
        if (lastj1 < 0) mma_commit(&sm.q_empty[1]);
        int pv_item[2] = {0, 0};  // this item's P V products per query tile (the first overwrites O)
        // Every K and V load phase is waited for, in order, whether or not a query tile uses the
        // key tile, so a stage is never refilled while its previous load could still be landing.
        auto wait_k = [&](int j) {
          const int p = kbase + j;
          return mbar_wait(&sm.k_full[p % NSK], (p / NSK) & 1, wait_ns);
        };
        auto wait_v = [&](int j) {
          const int p = kbase + j;
          return mbar_wait(&sm.v_full[p % NSV], (p / NSV) & 1, wait_ns);
        };
        // S_i(j): scores of query tile i against key tile j into TMEM columns [128 i, 128 i + 128).
        auto issue_s = [&](int i, int j) {
          tc_fence_after();
          const uint64_t qd = desc_add(qd0, i * 2 * QHALF);
          const uint64_t kd = desc_add(kd0, ((kbase + j) % NSK) * 2 * KHALF);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + 128 * i, desc_add(qd, (kk >> 2) * QHALF + (kk & 3) * 32),
                   desc_add(kd, (kk >> 2) * KHALF + (kk & 3) * 32), idesc_s, kk != 0);
          mma_commit(&sm.s_full[i]);
          if (j == (i ? lastj1 : lastj0)) mma_commit(&sm.q_empty[i]);
        };
        // O_i += P_i(j) V_j, P_i read from the first 64 columns of S_i.
        auto issue_pv = [&](int i, int j) -> bool {
          if (!mbar_wait(&sm.p_full[i], n_pv[i] & 1, wait_ns)) return false;
          tc_fence_after();
          const uint64_t vd = desc_add(vd0, ((kbase + j) % NSV) * 2 * KHALF);
          const uint32_t acc0 = pv_item[i] != 0;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + 256 + 128 * i, tmem + 128 * i + kk * 8, desc_add(vd, kk * 2048), idesc_pv,
                   kk == 0 ? acc0 : 1u);
          mma_commit(&sm.pv_done[i]);
          ++n_pv[i];
          ++pv_item[i];
          return true;
        };
        TileCursor cur(pl);
        int kt_next = n > 0 ? cur.seek(pl, 0) : 0;
        if (n > 0) {
          if (!wait_k(0)) { ok = false; break; }
          for (int i = 0; i < 2; ++i)
            if (rel(i, kt_next)) issue_s(i, 0);
          mma_commit(&sm.k_empty[kbase % NSK]);
        }
        for (int j = 0; ok && j < n; ++j) {
          const int kt = kt_next;
          const bool more = j + 1 < n;
          kt_next = more ? cur.seek(pl, j + 1) : 0;
          if (!wait_v(j)) { ok = false; break; }
          bool k_ready = !more;
          for (int i = 0; ok && i < 2; ++i) {
            if (rel(i, kt) && !issue_pv(i, j)) { ok = false; break; }
            if (more && rel(i, kt_next)) {
              if (!k_ready && !(k_ready = wait_k(j + 1))) { ok = false; break; }
              issue_s(i, j + 1);
            }
          }
          if (!ok) break;
          if (!k_ready && !wait_k(j + 1)) { ok = false; break; }
          // A stage is free once every product issued so far has completed: V_j after both P V
          // products of key tile j, K_{j+1} after both score products of key tile j + 1.
          mma_commit(&sm.v_empty[(kbase + j) % NSV]);
          if (more) mma_commit(&sm.k_empty[(kbase + j + 1) % NSK]);
        }
        if (!ok) break;
        kbase += n;
        mbar_arrive(&sm.item_empty[slot]);
      }
      if (!ok) fail(PG_ERR_TIMEOUT);
      // Every MMA issued above completes before TMEM is released.
      mma_commit(&sm.mma_done);
      mbar_wait(&sm.mma_done, 0, wait_ns);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax ----------
    const int i = (warp - 2) >> 2;                // query tile of this warpgroup
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;            // query row within the tile
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + 128 * i + lane_addr, t_o = tmem + 256 + 128 * i + lane_addr;
    int cs = 0;                                   // S_i products consumed, over all items
    const bool o_al32 = (reinterpret_cast<uintptr_t>(o) & 31) == 0;
    bool ok = true;
    for (uint32_t kq = 0; ok; ++kq) {
      const int slot = kq & 1;
      if (!warp_wait(&sm.item_full[slot], (kq >> 1) & 1, wait_ns)) { ok = false; break; }
      const Item& it = sm.item[slot];
      if (it.x < 0) break;
      const FwdTile tl = it.tl;
      const int h = it.h;
      const Plan& pl = it.plan;
      const int n = pl.n, n_a = pl.n_a;
      const int qlast = pl.last[i];
      auto rel = [&](int kt) { return qlast >= 0 && kt <= qlast; };
      const int row = tl.q0 + i * BM + r;
      const bool active = qlast >= 0;
      const bool valid = active && row <= qlast;
      const int rowc = valid ? row : (active ? qlast : tl.q0);
      const int4 ti = tok[rowc];                  // {g0, pe, own_lo, pos}
      const int first_row = tl.q0 + i * BM;
      float m_used = -INFINITY, l = 0.f;
      int c = 0;                                  // key tiles of this item done
      TileCursor cur(pl);
      for (int j = 0; active && j < n; ++j) {
        const int kt = cur.seek(pl, j);
        const int hi = cur.hi;
        if (!rel(kt)) continue;
        if (!warp_wait(&sm.s_full[i], cs & 1, wait_ns)) { ok = false; break; }
        tc_fence_after();
        // The row is handled 64 columns at a time (64 score registers).  Exact path (the first
        // key tile, or a tile whose max grows past the rescale threshold): the max of columns
        // 64..127 first (values dropped), then columns 0..63 (max, exp2, P), then 64..127 again
        // (exp2, P).  P of columns [32 h, 32 h + 32) goes to TMEM columns [16 h, 16 h + 16), over
        // scores this thread has already read.  Masked columns become -inf, so their P is exactly
        // zero; within one key tile a row's visible keys are one contiguous run of columns: in the
        // prefix range [kt, min(hi, row + 1)); in the responses' range the same run starting no
        // earlier than the row's own response (prefix rows get an empty run there).
        const bool full_tile = (j < n_a) && (kt + BN <= hi) && (kt + BN - 1 <= first_row);
        const int lo = (j < n_a) ? 0 : max(ti.z - kt, 0);
        const int len = max(min(hi, rowc + 1) - kt - lo, 0);
        uint32_t sr[64];
        bool stored = false;
        if (c > 0) {
          // Steady state: both halves straight to P with the running reference, the tile's max
          // tracked on the way; P is stored only if no row of the warp needs a rescale (then the
          // values are exactly those of the path below, which S, still intact, is rerun through).
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
            corr = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - m_new);
            m_used = m_new;
            l *= corr;
          }
          const float mref = (m_used == -INFINITY) ? 0.f : m_used;
          // Rescaling O needs the previous key tile's P V product done (it is: its S completed after
          // it, and a commit covers every earlier product; the wait returns at once).
          const bool any_rescale = __any_sync(0xffffffffu, rescale) && c > 0;
          if (any_rescale) {
            if (!warp_wait(&sm.pv_done[i], (cs - 1) & 1, wait_ns)) { ok = false; break; }
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
        ++cs;
        if (debug & PG_DEBUG_WITHHOLD_P) continue;   // test hook: never signal P (bounded waits)
        tc_fence_before();
        warp_arrive(&sm.p_full[i]);
      }
      // Epilogue: O / l and the natural-log LSE.
      if (active && ok && c > 0 && warp_wait(&sm.pv_done[i], (cs - 1) & 1, wait_ns)) {
        tc_fence_after();
        const float inv = 1.f / l;
        __nv_bfloat16* orow = o + ((size_t)rowc * Hq + h) * D;
#pragma unroll 1
        for (int q4 = 0; q4 < 4; ++q4) {
          uint32_t orr[32];
          tmem_ld32(t_o + q4 * 32, orr);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int e = 0; e < 32; e += 16) {
              uint32_t w[8];
#pragma unroll
              for (int u = 0; u < 8; ++u)
                w[u] = pack_bf16x2(__uint_as_float(orr[e + 2 * u]) * inv,
                                   __uint_as_float(orr[e + 2 * u + 1]) * inv);
              // 32-byte stores when o is 32-byte aligned (rows are 256 bytes apart), else 16-byte
              if (o_al32) {
                st_global_v8(orow + q4 * 32 + e, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
              } else {
                *reinterpret_cast<uint4*>(orow + q4 * 32 + e) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(orow + q4 * 32 + e + 8) = make_uint4(w[4], w[5], w[6], w[7]);
              }
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
      // This warp is done with the item (its O columns are read: the next item's first P V
      // product, which overwrites them, waits for this warpgroup's next P).
      tc_fence_before();
      warp_arrive(&sm.item_empty[slot]);
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
  // CTAs in chunks of query heads covering a few whole KV heads (about eight query heads).
  const int rep = a.Hq / a.Hkv;
  const int hc = order_chunk(a.Hkv, rep) * rep;
  prof_begin(PG_KERNEL_ATTN_FWD, a.stream);
  attn_fwd_sm100_kernel<<<(unsigned)(L->n_tiles[FWD256] * a.Hq), NTHREADS, smem, a.stream>>>(
      tq, tk, tv, static_cast<__nv_bfloat16*>(o), lse, tokens(L), tiles<FwdTile>(L, FWD256),
      intervals(L), lse2_out, padded_tokens(L), a.Hq, a.Hkv, (int)T, a.scale * kLog2e, hc,
      wait_ns, a.debug);
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
