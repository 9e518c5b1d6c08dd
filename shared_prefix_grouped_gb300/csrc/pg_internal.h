// Internal declarations shared by the host API and the kernels of the grouped-attention library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/pg_grouped_attn.h"
#include "../../include/pg_layer.h"

namespace pg {

// Work item of the forward and of the query-major dQ: query rows [q0, q1) of one group (tree).
// Its keys lie in "causal" ranges -- [g0, p_end) and a_cnt more ranges, entries a_off .. of the
// layout's interval table (the further ancestors of a nested prefix) -- in which row t sees key s
// iff s <= t, and in the "own" range [s_lo, s_hi), in which row t sees s iff own_lo(t) <= s <= t.
// For a two-level group [P; R1; ...; RG]: [g0, p_end) is the prefix (p_end = min(pe, q1)), the own
// range covers the tile's responses, a_cnt = 0.
struct FwdTile {
  int32_t q0, q1;      // query rows
  int32_t g0, p_end;   // first causal key range
  int32_t s_lo, s_hi;  // own key range (empty when the tile has no such rows)
  int32_t a_off, a_cnt;  // further causal ranges in the interval table
};

// The key ranges of a FwdTile in visiting order: causal ranges first, then the own range.
constexpr int kMaxKeyRanges = 8;
struct KeyRanges {
  int n, n_causal;
  int lo[kMaxKeyRanges], hi[kMaxKeyRanges];
  __host__ __device__ void init(const FwdTile& t, const int2* intervals) {
    n = 0;
    if (t.p_end > t.g0) {
      lo[n] = t.g0;
      hi[n] = t.p_end;
      ++n;
    }
    for (int i = 0; i < t.a_cnt && n < kMaxKeyRanges - 1; ++i) {
      const int2 iv = intervals[t.a_off + i];
      if (iv.y > iv.x) {
        lo[n] = iv.x;
        hi[n] = iv.y;
        ++n;
      }
    }
    n_causal = n;
    if (t.s_hi > t.s_lo) {
      lo[n] = t.s_lo;
      hi[n] = t.s_hi;
      ++n;
    }
  }
};

// Work item of the key-major backward: key rows [k0, k1) of one group and the query rows
// [q_lo, q_hi) that can see any of them (the rest of the prefix and every response of the group
// for a prefix key; the rest of the key's own response otherwise).
struct BwdTile {
  int32_t k0, k1;
  int32_t q_lo, q_hi;
  int32_t g0, pe;
  int32_t pad0, pad1;
};

static_assert(sizeof(FwdTile) == 32, "FwdTile layout");
static_assert(sizeof(BwdTile) == 32, "BwdTile layout");

// SPANS: one FwdTile per group with response rows: q0 = pe, q1 = the group's end, g0, p_end = pe,
// s_lo = pe, s_hi = q1, pe.
enum TileList { FWD64 = 0, FWD128 = 1, BWD64 = 2, BWD128 = 3, FWD256 = 4, SPANS = 5, NUM_LISTS = 6 };

// Row stride (elements) of the per-head fp32 rows the backward keeps for LSE and rowsum(dO * O):
// T rounded up to a multiple of 4, so every row starts 16-byte aligned (a TMA requirement).
inline int64_t padded_tokens(const pg_layout* L) { return (L->total_tokens + 3) & ~int64_t(3); }

// Maximum number of further causal ranges of a tile (a nested prefix deeper than this is refused).
constexpr int kMaxExtraRanges = kMaxKeyRanges - 2;

inline const int2* intervals(const pg_layout* L) {
  return reinterpret_cast<const int2*>(static_cast<const char*>(L->tables) + L->off_intervals);
}

inline const int4* tokens(const pg_layout* L) {
  return reinterpret_cast<const int4*>(static_cast<const char*>(L->tables) + L->off_tokens);
}
template <typename Tile>
inline const Tile* tiles(const pg_layout* L, int which) {
  return reinterpret_cast<const Tile*>(static_cast<const char*>(L->tables) + L->off_tiles[which]);
}

// CTA order of a grid of n_tiles x H work items (tile, head): heads in chunks of `hc` (the last
// chunk may be smaller); within a chunk the tiles run heaviest first (the lists are sorted) with the
// chunk's heads side by side.  A wave then touches the K/V or Q/dO rows of a few heads only, which
// stay in L2 while every tile of those heads streams them, and the grid still ends on light tiles.
__host__ __device__ inline void chunked_order(int x, int n_tiles, int H, int hc, int& tile,
                                              int& head) {
  const int full = H / hc;                      // complete chunks
  const int per_chunk = hc * n_tiles;
  if (x < full * per_chunk) {
    const int c = x / per_chunk, r = x - c * per_chunk;
    tile = r / hc;
    head = c * hc + r % hc;
  } else {
    const int hl = H - full * hc, r = x - full * per_chunk;
    tile = r / hl;
    head = full * hc + r % hl;
  }
}

// Heads per chunk for chunked_order: about eight query heads' worth of rows.
inline int order_chunk(int heads, int q_heads_per_head) {
  const int hc = 8 / (q_heads_per_head > 0 ? q_heads_per_head : 1);
  return hc < 1 ? 1 : (hc > heads ? heads : hc);
}

// Arguments common to every attention kernel launch.
struct AttnArgs {
  const pg_layout* layout;
  pg_dtype dtype;
  int Hq, Hkv, d;
  float scale;        // softmax scale
  float theta;        // RoPE base, 0 = off
  uint32_t flags, debug;
  cudaStream_t stream;
};

void set_error(const char* fmt, ...);

// Profiling hook (pg_set_profile): call before / after every kernel launch.
extern thread_local pg_profile* g_profile;
inline void prof_begin(pg_kernel kid, cudaStream_t s) {
  if (!g_profile) return;
  ++g_profile->launches;
  if (g_profile->kernel == kid && g_profile->ev_begin)
    cudaEventRecord(static_cast<cudaEvent_t>(g_profile->ev_begin), s);
}
inline void prof_end(pg_kernel kid, cudaStream_t s) {
  if (g_profile && g_profile->kernel == kid && g_profile->ev_end)
    cudaEventRecord(static_cast<cudaEvent_t>(g_profile->ev_end), s);
}
// Reads (and optionally clears) the device status words of every kernel file; first error wins.
pg_status read_kernel_status(bool clear, int32_t* code);
pg_status read_status_simt(bool clear, int32_t* code);
pg_status read_status_gemm(bool clear, int32_t* code);
pg_status read_status_fwd_sm100(bool clear, int32_t* code);
pg_status read_status_bwd_sm100(bool clear, int32_t* code);

// Tensor-core kernels (pg_attn_*_sm100.cu).
bool fwd_sm100_supported(const AttnArgs& a);
// lse2_out ([Hq][padded T], log2 units) is optional: a forward whose workspace the backward
// reuses writes the backward's copy of the LSE rows.
pg_status launch_fwd_sm100(const AttnArgs& a, const void* q, const void* k, const void* v, void* o,
                           float* lse, float* lse2_out = nullptr);
bool bwd_sm100_supported(const AttnArgs& a);
// dq_acc == nullptr: dK and dV only.
pg_status launch_bwd_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                           const void* dO, const float* lse2, const float* Dbuf, float* dq_acc,
                           void* dk, void* dv, const float2* rope_tab);
pg_status cuda_check(cudaError_t e, const char* what);

// Query-major dQ (pg_attn_dq_sm100.cu): dq (bf16, inverse-rotated with rope_tab when given) from
// the rotated q/k, v, dO and the preprocess's LSE_2 / Dsum rows.
bool dq_sm100_supported(const AttnArgs& a);
pg_status launch_dq_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                          const void* dO, const float* lse2, const float* Dbuf, void* dq,
                          const float2* rope_tab);
pg_status read_status_dq_sm100(bool clear, int32_t* code);

// Responses-only forward (pg_attn_score_sm100.cu): its launch shape and partial-result buffers.
struct ScorePlan {
  int hp;              // query heads per key/value head, packed into one CTA's rows
  int TB;              // tokens per row block (256 / hp)
  int nrb;             // row blocks per response span (the largest span decides)
  int nsplit;          // prefix-key splits per row block
  int64_t nblk;        // CTAs per split: spans x nrb x Hkv
  size_t part_o_bytes, part_lse_bytes;   // fp32 partials (0 when nsplit == 1)
};
bool score_sm100_supported(const AttnArgs& a);
ScorePlan score_plan(const pg_layout* L, int Hq, int Hkv);
pg_status launch_score_sm100(const AttnArgs& a, const void* q, const void* k, const void* v,
                             void* o, float* lse, float* part_o, float* part_lse);
pg_status read_status_score_sm100(bool clear, int32_t* code);

// RoPE frequencies inv_freq_k = theta^(-2k/d), k < d/2 (computed on the host in fp64), as
// fractions of a turn: turn[k] = frac(inv_freq_k / 2 pi) in 0.64 fixed point, so that position x
// turn[k] taken modulo 2^64 is the angle already reduced to one turn (integer arithmetic in the
// kernel: double precision is slow on this part).
struct RopeFreq {
  uint64_t turn[64];
};

// Which token rows a RoPE pass rotates: every row of both tensors, or every row of the first
// tensor and only the response rows (the layout's response spans) of the second, in separate
// blocks of one launch.
enum class RopeRows { kAll, kAllThenResponses };

// SIMT kernels (pg_simt.cu).
pg_status launch_rope(const AttnArgs& a, const void* x0, void* y0, int heads0, const void* x1,
                      void* y1, int heads1, bool inverse, bool in_fp32, float2* table_out,
                      const float2* table_in, RopeRows rows = RopeRows::kAll);
pg_status launch_fwd_simt(const AttnArgs& a, const void* q, const void* k, const void* v, void* o,
                          float* lse);
pg_status launch_bwd_simt(const AttnArgs& a, const void* q, const void* k, const void* v,
                          const void* o, const float* lse, const void* dO, float* Dbuf,
                          float* dq_acc, float* dk_acc, void* dv);
// Padded layouts: zero the padding rows of up to three [T, heads, d] tensors of the call's dtype
// and, with lse, set lse[h][row] = +inf on them.
pg_status launch_pad_fill(const AttnArgs& a, void* x0, int heads0, void* x1, int heads1, void* x2,
                          int heads2, float* lse);
// dq_acc may be nullptr (nothing to zero); lse2_ready: the forward already wrote lse2's rows.
pg_status launch_bwd_preprocess(const AttnArgs& a, const void* o, const void* dO, const float* lse,
                                float* Dbuf, float* lse2, float* dq_acc, bool lse2_ready = false);

}  // namespace pg
