// Host side of the grouped-attention C ABI: packing, argument checks, workspace, dispatch.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <numeric>
#include <vector>

#include "pg_internal.h"

namespace pg {

static thread_local char g_msg[512] = "";
thread_local pg_profile* g_profile = nullptr;

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

pg_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return PG_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return PG_ERR_CUDA;
}

static int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

pg_status read_kernel_status(bool clear, int32_t* code) {
  *code = 0;
  pg_status st = read_status_simt(clear, code);
  if (st == PG_OK) st = read_status_gemm(clear, code);
  if (st == PG_OK) st = read_status_fwd_sm100(clear, code);
  if (st == PG_OK) st = read_status_bwd_sm100(clear, code);
  if (st == PG_OK) st = read_status_score_sm100(clear, code);
  if (st == PG_OK) st = read_status_dq_sm100(clear, code);
  return st;
}

// ---------------------------------------------------------------------------------------------
// Packing.  Groups are laid out back to back; within a group the prefix is followed by its
// responses ("Sequential Concatenation" of the skill page; [P; R1; ...; RG] of the Pith review).
// ---------------------------------------------------------------------------------------------

struct Plan {
  int64_t T = 0, segs = 0, max_pos = 0, pairs = 0;
  int64_t n[NUM_LISTS] = {0, 0, 0, 0, 0, 0};
  int64_t off[NUM_LISTS] = {0, 0, 0, 0, 0, 0};
  int64_t off_tokens = 0, bytes = 0;
  int64_t max_resp = 0;   // largest number of response rows in one group
  int64_t n_pad = 0, off_pad = 0;   // padded layouts: padding-row list
  int64_t max_depth = 0;            // segments on the longest root-to-leaf path
  int64_t n_iv = 0, off_iv = 0;     // interval table of the tiles' further causal ranges
};

static pg_status check_lengths(int32_t B, const int32_t* lp, const int32_t* gs, const int32_t* rs,
                               Plan* p) {
  if (B < 1 || !lp || !gs) {
    set_error("pg_pack: num_groups must be >= 1 and arrays non-NULL");
    return PG_ERR_INVALID_ARG;
  }
  int64_t T = 0, S = 0, maxpos = 0, pairs = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (lp[b] < 0 || gs[b] < 0) {
      set_error("pg_pack: negative prefix length or group size in group %d", b);
      return PG_ERR_INVALID_ARG;
    }
    int64_t L = lp[b];
    T += L;
    maxpos = std::max(maxpos, L);
    pairs += L * (L + 1) / 2;
    if (gs[b] > 0 && !rs) {
      set_error("pg_pack: suffix_lens is NULL");
      return PG_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < gs[b]; ++i, ++S) {
      int64_t r = rs[S];
      if (r < 0) {
        set_error("pg_pack: negative suffix length at response %lld", (long long)S);
        return PG_ERR_INVALID_ARG;
      }
      T += r;
      maxpos = std::max(maxpos, L + r);
      pairs += r * L + r * (r + 1) / 2;
      if (T >= (int64_t(1) << 30)) break;
    }
    if (T >= (int64_t(1) << 30)) break;
  }
  if (T <= 0 || T >= (int64_t(1) << 30)) {
    set_error("pg_pack: total tokens must be in [1, 2^30), got %lld", (long long)T);
    return PG_ERR_INVALID_ARG;
  }
  p->T = T;
  p->segs = S;
  p->max_pos = maxpos;
  p->pairs = pairs;
  // Work-list lengths: one tile per started block of rows in each group.
  int64_t n64 = 0, n128 = 0, n256 = 0, nspan = 0;
  int64_t s = 0;
  for (int32_t b = 0; b < B; ++b) {
    int64_t resp = 0;
    for (int32_t i = 0; i < gs[b]; ++i) resp += rs[s++];
    const int64_t len = lp[b] + resp;
    n64 += (len + 63) / 64;
    n128 += (len + 127) / 128;
    n256 += (len + 255) / 256;
    nspan += resp > 0;
    p->max_resp = std::max(p->max_resp, resp);
    p->max_depth = std::max<int64_t>(p->max_depth, (gs[b] > 0 && lp[b] > 0) ? 2 : 1);
  }
  p->n[FWD64] = p->n[BWD64] = n64;
  p->n[FWD128] = p->n[BWD128] = n128;
  p->n[FWD256] = n256;
  p->n[SPANS] = nspan;
  int64_t off = 0;
  p->off_tokens = off;
  off = align_up(off + 16 * T, 256);
  for (int w = 0; w < NUM_LISTS; ++w) {
    p->off[w] = off;
    off = align_up(off + 32 * p->n[w], 256);
  }
  p->off_iv = off;    // two-level tiles need no further ranges: empty table
  p->bytes = off;
  return PG_OK;
}

template <typename Tile>
static void sort_by_cost(std::vector<Tile>& v, std::vector<int64_t>& cost) {
  std::vector<size_t> idx(v.size());
  std::iota(idx.begin(), idx.end(), 0);
  std::stable_sort(idx.begin(), idx.end(), [&](size_t a, size_t b) { return cost[a] > cost[b]; });
  std::vector<Tile> out(v.size());
  for (size_t i = 0; i < idx.size(); ++i) out[i] = v[idx[i]];
  v.swap(out);
}

static void build_tables(int32_t B, const int32_t* lp, const int32_t* gs, const int32_t* rs,
                         const Plan& p, int32_t* pos, char* tables) {
  int4* tok = reinterpret_cast<int4*>(tables + p.off_tokens);
  std::vector<int32_t> seg_end_of(p.T);  // row after the token's own response (or group end)
  int32_t row = 0;
  int64_t s = 0;
  for (int32_t b = 0; b < B; ++b) {
    int32_t g0 = row, pe = row + lp[b];
    for (int32_t j = 0; j < lp[b]; ++j, ++row) {
      tok[row] = make_int4(g0, pe, g0, j);
      pos[row] = j;
      seg_end_of[row] = pe;
    }
    for (int32_t i = 0; i < gs[b]; ++i, ++s) {
      int32_t own = row;
      for (int32_t j = 0; j < rs[s]; ++j, ++row) {
        tok[row] = make_int4(g0, pe, own, lp[b] + j);
        pos[row] = lp[b] + j;
        seg_end_of[row] = own + rs[s];
      }
    }
  }
  // Work lists, per group, for 64-, 128- and 256-row tiles (no key-major list for 256); heaviest
  // first.
  for (int bm = 64, wi = 0; bm <= 256; bm *= 2, ++wi) {
    std::vector<FwdTile> ft;
    std::vector<BwdTile> bt;
    std::vector<int64_t> fc, bc;
    int32_t g0 = 0;
    int64_t sb = 0;
    for (int32_t b = 0; b < B; ++b) {
      int32_t pe = g0 + lp[b];
      int32_t gend = pe;
      for (int32_t i = 0; i < gs[b]; ++i) gend += rs[sb + i];
      sb += gs[b];
      if (gend == g0) continue;
      for (int32_t q0 = g0; q0 < gend; q0 += bm) {
        int32_t q1 = std::min(q0 + bm, gend);
        FwdTile t{};
        t.q0 = q0;
        t.q1 = q1;
        t.g0 = g0;
        t.p_end = std::min(pe, q1);
        if (q1 > pe) {
          t.s_lo = tok[std::max(q0, pe)].z;
          t.s_hi = q1;
        } else {
          t.s_lo = t.s_hi = q1;
        }
        ft.push_back(t);
        fc.push_back(int64_t(q1 - q0) * ((t.p_end - g0) + (t.s_hi - t.s_lo)));
        BwdTile u{};
        u.k0 = q0;
        u.k1 = q1;
        u.g0 = g0;
        u.pe = pe;
        u.q_lo = q0;
        u.q_hi = (q0 < pe) ? gend : seg_end_of[q1 - 1];
        bt.push_back(u);
        bc.push_back(int64_t(q1 - q0) * (u.q_hi - u.q_lo));
      }
      g0 = gend;
    }
    sort_by_cost(ft, fc);
    sort_by_cost(bt, bc);
    const int fw = wi == 0 ? FWD64 : wi == 1 ? FWD128 : FWD256;
    memcpy(tables + p.off[fw], ft.data(), ft.size() * sizeof(FwdTile));
    if (wi < 2) {
      const int bw = wi == 0 ? BWD64 : BWD128;
      memcpy(tables + p.off[bw], bt.data(), bt.size() * sizeof(BwdTile));
    }
  }
  // Response spans, in group order.
  std::vector<FwdTile> spans;
  int32_t g0 = 0;
  int64_t sb = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t pe = g0 + lp[b];
    int32_t gend = pe;
    for (int32_t i = 0; i < gs[b]; ++i) gend += rs[sb + i];
    sb += gs[b];
    if (gend > pe) {
      FwdTile t{};
      t.q0 = pe;
      t.q1 = gend;
      t.g0 = g0;
      t.p_end = pe;
      t.s_lo = pe;
      t.s_hi = gend;
      spans.push_back(t);
    }
    g0 = gend;
  }
  memcpy(tables + p.off[SPANS], spans.data(), spans.size() * sizeof(FwdTile));
}

// Padded layouts: the same plan as packing every slot at its full length, plus the list of
// padding rows appended to the tables.
struct Padded {
  std::vector<int32_t> lp, gs, rs;
  const int32_t* rlen = nullptr;
  int32_t R = 0;
};

static pg_status plan_padded(int32_t B, int32_t Lp, int32_t G, int32_t R, const int32_t* rlen,
                             Padded* pd, Plan* p) {
  if (B < 1 || Lp < 0 || G < 0 || R < 0 || (G > 0 && R > 0 && !rlen)) {
    set_error("pg_pack_padded: num_groups >= 1, lengths >= 0 and response_lens non-NULL required");
    return PG_ERR_INVALID_ARG;
  }
  int64_t n_pad = 0;
  for (int64_t i = 0; i < (int64_t)B * G; ++i) {
    const int32_t r = R > 0 ? rlen[i] : 0;
    if (r < 0 || r > R) {
      set_error("pg_pack_padded: response %lld has length %d outside [0, %d]", (long long)i, r, R);
      return PG_ERR_INVALID_ARG;
    }
    n_pad += R - r;
  }
  pd->lp.assign(B, Lp);
  pd->gs.assign(B, G);
  pd->rs.assign((size_t)B * G, R);
  pd->rlen = rlen;
  pd->R = R;
  pg_status st = check_lengths(B, pd->lp.data(), pd->gs.data(), pd->rs.data(), p);
  if (st != PG_OK) return st;
  p->n_pad = n_pad;
  p->off_pad = p->bytes;
  p->bytes = align_up(p->bytes + 4 * n_pad, 256);
  return PG_OK;
}

static void build_pad_list(int32_t B, int32_t Lp, int32_t G, const Padded& pd, const Plan& p,
                           char* tables) {
  int32_t* out = reinterpret_cast<int32_t*>(tables + p.off_pad);
  int64_t row = 0, n = 0;
  for (int32_t b = 0; b < B; ++b) {
    row += Lp;
    for (int32_t i = 0; i < G; ++i, row += pd.R) {
      const int32_t r = pd.R > 0 ? pd.rlen[(int64_t)b * G + i] : 0;
      for (int32_t j = r; j < pd.R; ++j) out[n++] = (int32_t)(row + j);
    }
  }
}

static void fill_layout(int32_t B, const Plan& p, const int32_t* pos, const void* tables,
                        pg_layout* L) {
  memset(L, 0, sizeof(*L));
  L->num_groups = B;
  L->num_segments = p.segs;
  L->total_tokens = p.T;
  L->max_position = p.max_pos;
  L->pairs = p.pairs;
  for (int w = 0; w < NUM_LISTS; ++w) {
    L->n_tiles[w] = p.n[w];
    L->off_tiles[w] = p.off[w];
  }
  L->off_tokens = p.off_tokens;
  L->table_bytes = p.bytes;
  L->position_ids = pos;
  L->tables = tables;
  L->max_response_rows = p.max_resp;
  L->n_pad_rows = p.n_pad;
  L->off_pad_rows = p.off_pad;
  L->max_depth = p.max_depth;
  L->n_intervals = p.n_iv;
  L->off_intervals = p.off_iv;
}

// ---------------------------------------------------------------------------------------------
// Nested prefixes (trees).  Segments are listed in depth-first preorder, parent before child; the
// packed rows follow that order, so every node's subtree is one contiguous row range.  A token sees
// all tokens of its node's ancestors and its own node's tokens up to itself; its position is the
// total length of its ancestors plus its offset in its node (its position in the root-to-leaf
// sequence the repeated-prefix baseline would run).
// ---------------------------------------------------------------------------------------------

struct Tree {
  std::vector<int32_t> parent, len, start, end, sub_end, off, depth, root_start, root_end;
  std::vector<char> leaf;
  // Work units: a single node, or a run of consecutive sibling leaves.
  struct Unit {
    int32_t r0, r1;        // rows
    int32_t node;          // the node (single-node unit) or the leaves' parent
    bool run;
  };
  std::vector<Unit> units;
};

static pg_status plan_tree(int32_t N, const int32_t* parent, const int32_t* len, Tree* tr,
                           Plan* p) {
  if (N < 1 || !parent || !len) {
    set_error("pg_pack_tree: num_nodes must be >= 1 and arrays non-NULL");
    return PG_ERR_INVALID_ARG;
  }
  tr->parent.assign(parent, parent + N);
  tr->len.assign(len, len + N);
  tr->start.resize(N);
  tr->end.resize(N);
  tr->sub_end.resize(N);
  tr->off.resize(N);
  tr->depth.resize(N);
  tr->root_start.resize(N);
  tr->root_end.resize(N);
  tr->leaf.assign(N, 1);
  std::vector<int32_t> stack;
  int64_t row = 0, pairs = 0, maxpos = 0, maxdepth = 0;
  for (int32_t i = 0; i < N; ++i) {
    const int32_t par = parent[i];
    if (len[i] < 0 || par < -1 || par >= i) {
      set_error("pg_pack_tree: node %d has a negative length or a parent not listed before it", i);
      return PG_ERR_INVALID_ARG;
    }
    // Depth-first preorder: the parent must be on the current root-to-node path.
    while (!stack.empty() && stack.back() != par) {
      tr->sub_end[stack.back()] = (int32_t)row;
      stack.pop_back();
    }
    if (par >= 0 && stack.empty()) {
      set_error("pg_pack_tree: node %d does not follow its parent's subtree in depth-first order",
                i);
      return PG_ERR_INVALID_ARG;
    }
    tr->start[i] = (int32_t)row;
    row += len[i];
    tr->end[i] = (int32_t)row;
    if (par >= 0) {
      tr->leaf[par] = 0;
      tr->off[i] = tr->off[par] + len[par];
      tr->depth[i] = tr->depth[par] + 1;
      tr->root_start[i] = tr->root_start[par];
      tr->root_end[i] = tr->root_end[par];
    } else {
      tr->off[i] = 0;
      tr->depth[i] = 1;
      tr->root_start[i] = tr->start[i];
      tr->root_end[i] = tr->end[i];
    }
    pairs += (int64_t)len[i] * tr->off[i] + (int64_t)len[i] * (len[i] + 1) / 2;
    maxpos = std::max<int64_t>(maxpos, (int64_t)tr->off[i] + len[i]);
    maxdepth = std::max<int64_t>(maxdepth, tr->depth[i]);
    if (row >= (int64_t(1) << 30)) break;
    stack.push_back(i);
  }
  while (!stack.empty()) {
    tr->sub_end[stack.back()] = (int32_t)row;
    stack.pop_back();
  }
  if (row <= 0 || row >= (int64_t(1) << 30)) {
    set_error("pg_pack_tree: total tokens must be in [1, 2^30), got %lld", (long long)row);
    return PG_ERR_INVALID_ARG;
  }
  if (maxdepth > kMaxExtraRanges + 2) {
    set_error("pg_pack_tree: nesting depth %lld exceeds %d", (long long)maxdepth,
              kMaxExtraRanges + 2);
    return PG_ERR_UNSUPPORTED;
  }
  // Units: runs of consecutive sibling leaves (non-root), else single nodes; empty nodes skipped.
  for (int32_t i = 0; i < N; ++i) {
    if (len[i] == 0) continue;
    const bool run = tr->leaf[i] && parent[i] >= 0;
    if (run && !tr->units.empty() && tr->units.back().run && tr->units.back().node == parent[i] &&
        tr->units.back().r1 == tr->start[i]) {
      tr->units.back().r1 = tr->end[i];
      continue;
    }
    tr->units.push_back({tr->start[i], tr->end[i], run ? parent[i] : i, run});
  }
  int64_t roots = 0;
  for (int32_t i = 0; i < N; ++i) roots += parent[i] < 0;
  p->T = row;
  p->segs = N;
  p->max_pos = maxpos;
  p->pairs = pairs;
  p->max_depth = maxdepth;
  p->max_resp = 0;
  // Tile counts per unit; the interval table holds, per forward tile, the causal ranges beyond the
  // first (at most depth - 1 of them).
  int64_t n64 = 0, n128 = 0, n256 = 0, n_iv = 0;
  for (const auto& u : tr->units) {
    const int64_t L = u.r1 - u.r0;
    n64 += (L + 63) / 64;
    n128 += (L + 127) / 128;
    n256 += (L + 255) / 256;
    const int64_t extra = std::max<int64_t>(0, tr->depth[u.node] - 1);
    n_iv += extra * ((L + 63) / 64 + (L + 127) / 128 + (L + 255) / 256);
  }
  p->n[FWD64] = p->n[BWD64] = n64;
  p->n[FWD128] = p->n[BWD128] = n128;
  p->n[FWD256] = n256;
  // A tree of depth <= 2 is a two-level group: give it the response spans of the scoring path.
  int64_t nspan = 0;
  if (maxdepth <= 2)
    for (int32_t i = 0; i < N; ++i)
      if (parent[i] < 0 && tr->sub_end[i] > tr->end[i]) {
        ++nspan;
        p->max_resp = std::max<int64_t>(p->max_resp, tr->sub_end[i] - tr->end[i]);
      }
  p->n[SPANS] = nspan;
  p->n_iv = n_iv;
  int64_t off = 0;
  p->off_tokens = off;
  off = align_up(off + 16 * row, 256);
  for (int w = 0; w < NUM_LISTS; ++w) {
    p->off[w] = off;
    off = align_up(off + 32 * p->n[w], 256);
  }
  p->off_iv = off;
  off = align_up(off + 8 * n_iv, 256);
  p->bytes = off;
  (void)roots;
  return PG_OK;
}

static void build_tree_tables(const Tree& tr, const Plan& p, int32_t* pos, char* tables) {
  const int32_t N = (int32_t)tr.parent.size();
  int4* tok = reinterpret_cast<int4*>(tables + p.off_tokens);
  std::vector<int32_t> node_end(p.T);      // end of each row's own node
  for (int32_t i = 0; i < N; ++i)
    for (int32_t t = tr.start[i]; t < tr.end[i]; ++t) {
      const int32_t ps = tr.off[i] + (t - tr.start[i]);
      tok[t] = make_int4(tr.root_start[i], tr.root_end[i], tr.start[i], ps);
      pos[t] = ps;
      node_end[t] = tr.end[i];
    }
  int2* ivs = reinterpret_cast<int2*>(tables + p.off_iv);
  int64_t n_iv = 0;
  // The causal ranges a unit's query rows need: its node's ancestors (root first) and, for a
  // single-node unit, the node itself (clipped to the tile's last row).
  auto ancestors = [&](int32_t node, bool include_self, std::vector<int2>& out) {
    out.clear();
    for (int32_t a = include_self ? node : tr.parent[node]; a >= 0; a = tr.parent[a])
      if (tr.len[a] > 0) out.push_back(make_int2(tr.start[a], tr.end[a]));
    std::reverse(out.begin(), out.end());
  };
  std::vector<int2> anc;
  for (int bm = 64, wi = 0; bm <= 256; bm *= 2, ++wi) {
    std::vector<FwdTile> ft;
    std::vector<BwdTile> bt;
    std::vector<int64_t> fc, bc;
    for (const auto& u : tr.units) {
      ancestors(u.node, true, anc);   // the node itself, or the leaves' parent, and above
      int64_t anc_keys = 0;
      for (const auto& a : anc) anc_keys += a.y - a.x;
      for (int32_t q0 = u.r0; q0 < u.r1; q0 += bm) {
        const int32_t q1 = std::min(q0 + bm, u.r1);
        FwdTile t{};
        t.q0 = q0;
        t.q1 = q1;
        // First causal range: the outermost; the others go to the interval table.
        std::vector<int2> rng(anc);
        if (!u.run) rng.back().y = std::min(rng.back().y, q1);
        t.g0 = rng.empty() ? q0 : rng[0].x;
        t.p_end = rng.empty() ? q0 : rng[0].y;
        t.a_off = (int32_t)n_iv;
        t.a_cnt = (int32_t)(rng.size() > 0 ? rng.size() - 1 : 0);
        for (size_t k = 1; k < rng.size(); ++k) ivs[n_iv++] = rng[k];
        if (u.run) {
          t.s_lo = tok[q0].z;
          t.s_hi = q1;
        } else {
          t.s_lo = t.s_hi = q1;
        }
        ft.push_back(t);
        fc.push_back((int64_t)(q1 - q0) * (anc_keys + (t.s_hi - t.s_lo)));
        if (wi < 2) {
          // Key-major: keys [q0, q1) are seen by rows from themselves up to the end of their
          // node's subtree (a single node) or of their own leaf (a run of leaves).
          BwdTile b{};
          b.k0 = q0;
          b.k1 = q1;
          b.q_lo = q0;
          b.g0 = tok[q0].x;
          if (u.run) {
            b.q_hi = node_end[q1 - 1];
            b.pe = q0;             // every key of the tile is seen by its own leaf's rows only
          } else {
            b.q_hi = tr.sub_end[u.node];
            b.pe = q1;             // every key is seen by all later rows of the subtree
          }
          bt.push_back(b);
          bc.push_back((int64_t)(q1 - q0) * (b.q_hi - b.q_lo));
        }
      }
    }
    sort_by_cost(ft, fc);
    sort_by_cost(bt, bc);
    const int fw = wi == 0 ? FWD64 : wi == 1 ? FWD128 : FWD256;
    memcpy(tables + p.off[fw], ft.data(), ft.size() * sizeof(FwdTile));
    if (wi < 2) {
      const int bw = wi == 0 ? BWD64 : BWD128;
      memcpy(tables + p.off[bw], bt.data(), bt.size() * sizeof(BwdTile));
    }
  }
  if (p.n[SPANS] > 0) {
    std::vector<FwdTile> spans;
    for (int32_t i = 0; i < N; ++i)
      if (tr.parent[i] < 0 && tr.sub_end[i] > tr.end[i]) {
        FwdTile t{};
        t.q0 = tr.end[i];
        t.q1 = tr.sub_end[i];
        t.g0 = tr.start[i];
        t.p_end = tr.end[i];
        t.s_lo = tr.end[i];
        t.s_hi = tr.sub_end[i];
        spans.push_back(t);
      }
    memcpy(tables + p.off[SPANS], spans.data(), spans.size() * sizeof(FwdTile));
  }
}

// Copies a host-built layout to the caller's device buffers and points *layout at them.
static pg_status upload_layout(const std::vector<int32_t>& pos, const std::vector<char>& tab,
                               int32_t* position_ids_dev, void* tables_dev, const pg_layout& host,
                               pg_layout* layout, cudaStream_t s) {
  pg_status st = cuda_check(cudaMemcpyAsync(position_ids_dev, pos.data(), pos.size() * 4,
                                            cudaMemcpyHostToDevice, s),
                            "pg_pack: copy position ids");
  if (st != PG_OK) return st;
  st = cuda_check(cudaMemcpyAsync(tables_dev, tab.data(), tab.size(), cudaMemcpyHostToDevice, s),
                  "pg_pack: copy tables");
  if (st != PG_OK) return st;
  // Pageable-source copies return once the source has been staged; make that explicit so the
  // vectors can be released whatever the runtime's staging policy.
  st = cuda_check(cudaStreamSynchronize(s), "pg_pack: synchronize");
  if (st != PG_OK) return st;
  *layout = host;
  layout->position_ids = position_ids_dev;
  layout->tables = tables_dev;
  return PG_OK;
}

// ---------------------------------------------------------------------------------------------
// Attention argument checks and workspace
// ---------------------------------------------------------------------------------------------

struct WsPlan {
  size_t q_rot = 0, k_rot = 0, rope_tab = 0, Dbuf = 0, lse2 = 0, dq_acc = 0, dk_acc = 0;
  size_t part_o = 0, part_lse = 0, total = 0;
};

static size_t esize(pg_dtype dt) { return dt == PG_F32 ? 4 : 2; }

static WsPlan ws_plan(const pg_layout* L, pg_dtype dt, int Hq, int Hkv, int d, bool rope,
                      int phase, const AttnArgs& a) {
  WsPlan w;
  size_t T = (size_t)L->total_tokens;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = (size_t)align_up((int64_t)(off + bytes), 256);
    return o;
  };
  // Offset 0 is a valid slot; record "absent" as SIZE_MAX.
  w.q_rot = w.k_rot = w.rope_tab = w.Dbuf = w.lse2 = w.dq_acc = w.dk_acc = SIZE_MAX;
  w.part_o = w.part_lse = SIZE_MAX;
  if (rope && (a.flags & PG_FLAG_PRE_ROTATED)) {
    // q and k come rotated; only the backward's cos/sin table, at offset 0 (pg_rope_table).
    if (phase == 1) w.rope_tab = take(T * (d / 2) * sizeof(float2));
  } else if (rope) {
    w.q_rot = take(T * Hq * d * esize(dt));
    w.k_rot = take(T * Hkv * d * esize(dt));
    if (phase == 1) w.rope_tab = take(T * (d / 2) * sizeof(float2));
  }
  if (phase == 0 && (a.flags & PG_FLAG_RESPONSES_ONLY) && !(a.flags & PG_FLAG_SIMT) &&
      score_sm100_supported(a)) {
    const ScorePlan sp = score_plan(L, Hq, Hkv);
    if (sp.nsplit > 1) {
      w.part_o = take(sp.part_o_bytes);
      w.part_lse = take(sp.part_lse_bytes);
    }
  }
  if (phase == 1) {
    const size_t Tp = (size_t)padded_tokens(L);
    const bool sm100 = !(a.flags & PG_FLAG_SIMT) && bwd_sm100_supported(a);
    w.Dbuf = take(Tp * Hq * sizeof(float));
    w.lse2 = take(Tp * Hq * sizeof(float));
    // The query-major dQ kernel writes dq directly: no fp32 accumulator.
    if (!(sm100 && (a.flags & PG_FLAG_DETERMINISTIC) && dq_sm100_supported(a)))
      w.dq_acc = take(T * Hq * d * sizeof(float));
    if (!sm100) w.dk_acc = take(T * Hkv * d * sizeof(float));
  }
  w.total = off;
  return w;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static pg_status check_attn(const pg_layout* L, pg_dtype dt, int Hq, int Hkv, int d,
                            const pg_opts* opts, std::initializer_list<const void*> ptrs,
                            const char* who) {
  if (!L || !L->tables || !L->position_ids || L->total_tokens <= 0) {
    set_error("%s: layout missing or empty (call pg_pack first)", who);
    return PG_ERR_INVALID_ARG;
  }
  if (dt != PG_F32 && dt != PG_BF16) {
    set_error("%s: unknown dtype %d", who, (int)dt);
    return PG_ERR_INVALID_ARG;
  }
  if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0) {
    set_error("%s: heads_q (%d) must be a positive multiple of heads_kv (%d)", who, Hq, Hkv);
    return PG_ERR_INVALID_ARG;
  }
  if (d != 64 && d != 128) {
    set_error("%s: head_dim must be 64 or 128, got %d", who, d);
    return PG_ERR_INVALID_ARG;
  }
  if (opts && (opts->softmax_scale < 0.f || opts->rope_theta < 0.f)) {
    set_error("%s: softmax_scale and rope_theta must be >= 0", who);
    return PG_ERR_INVALID_ARG;
  }
  if (opts && (opts->flags & PG_FLAG_PRE_ROTATED) && !(opts->rope_theta > 0.f)) {
    set_error("%s: PG_FLAG_PRE_ROTATED needs rope_theta > 0", who);
    return PG_ERR_INVALID_ARG;
  }
  int i = 0;
  for (const void* p : ptrs) {
    if (!p || !aligned16(p)) {
      set_error("%s: pointer argument %d is NULL or not 16-byte aligned", who, i);
      return PG_ERR_INVALID_ARG;
    }
    ++i;
  }
  return PG_OK;
}

static AttnArgs make_args(const pg_layout* L, pg_dtype dt, int Hq, int Hkv, int d,
                          const pg_opts* opts, cudaStream_t s) {
  AttnArgs a;
  a.layout = L;
  a.dtype = dt;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.scale = (opts && opts->softmax_scale > 0.f) ? opts->softmax_scale : 1.0f / sqrtf((float)d);
  a.theta = opts ? opts->rope_theta : 0.f;
  a.flags = opts ? opts->flags : 0u;
  a.debug = opts ? opts->debug : 0u;
  a.stream = s;
  return a;
}

}  // namespace pg

using namespace pg;

extern "C" {

pg_status pg_pack_size(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                       const int32_t* suffix_lens, int64_t* total_tokens, int64_t* table_bytes) {
  Plan p;
  pg_status st = check_lengths(num_groups, prefix_lens, group_sizes, suffix_lens, &p);
  if (st != PG_OK) return st;
  if (total_tokens) *total_tokens = p.T;
  if (table_bytes) *table_bytes = p.bytes;
  return PG_OK;
}

pg_status pg_pack_host(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                       const int32_t* suffix_lens, int32_t* position_ids, void* tables,
                       int64_t table_bytes, pg_layout* layout) {
  Plan p;
  pg_status st = check_lengths(num_groups, prefix_lens, group_sizes, suffix_lens, &p);
  if (st != PG_OK) return st;
  if (!position_ids || !tables || !layout || table_bytes < p.bytes) {
    set_error("pg_pack_host: NULL buffer or table buffer smaller than %lld bytes",
              (long long)p.bytes);
    return PG_ERR_INVALID_ARG;
  }
  memset(tables, 0, (size_t)p.bytes);
  build_tables(num_groups, prefix_lens, group_sizes, suffix_lens, p, position_ids,
               static_cast<char*>(tables));
  fill_layout(num_groups, p, position_ids, tables, layout);
  return PG_OK;
}

pg_status pg_pack(int32_t num_groups, const int32_t* prefix_lens, const int32_t* group_sizes,
                  const int32_t* suffix_lens, int32_t* position_ids_dev, void* tables_dev,
                  int64_t table_bytes, pg_layout* layout, pg_stream_t stream) {
  Plan p;
  pg_status st = check_lengths(num_groups, prefix_lens, group_sizes, suffix_lens, &p);
  if (st != PG_OK) return st;
  if (!position_ids_dev || !tables_dev || !layout || table_bytes < p.bytes) {
    set_error("pg_pack: NULL buffer or table buffer smaller than %lld bytes", (long long)p.bytes);
    return PG_ERR_INVALID_ARG;
  }
  std::vector<int32_t> pos((size_t)p.T);
  std::vector<char> tab((size_t)p.bytes);
  pg_layout host;
  st = pg_pack_host(num_groups, prefix_lens, group_sizes, suffix_lens, pos.data(), tab.data(),
                    p.bytes, &host);
  if (st != PG_OK) return st;
  return upload_layout(pos, tab, position_ids_dev, tables_dev, host, layout,
                       reinterpret_cast<cudaStream_t>(stream));
}

pg_status pg_pack_tree_size(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                            int64_t* total_tokens, int64_t* table_bytes) {
  Plan p;
  Tree tr;
  pg_status st = plan_tree(num_nodes, parent, seg_lens, &tr, &p);
  if (st != PG_OK) return st;
  if (total_tokens) *total_tokens = p.T;
  if (table_bytes) *table_bytes = p.bytes;
  return PG_OK;
}

pg_status pg_pack_tree_host(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                            int32_t* position_ids, void* tables, int64_t table_bytes,
                            pg_layout* layout) {
  Plan p;
  Tree tr;
  pg_status st = plan_tree(num_nodes, parent, seg_lens, &tr, &p);
  if (st != PG_OK) return st;
  if (!position_ids || !tables || !layout || table_bytes < p.bytes) {
    set_error("pg_pack_tree_host: NULL buffer or table buffer smaller than %lld bytes",
              (long long)p.bytes);
    return PG_ERR_INVALID_ARG;
  }
  memset(tables, 0, (size_t)p.bytes);
  build_tree_tables(tr, p, position_ids, static_cast<char*>(tables));
  int32_t roots = 0;
  for (int32_t i = 0; i < num_nodes; ++i) roots += parent[i] < 0;
  fill_layout(roots, p, position_ids, tables, layout);
  return PG_OK;
}

pg_status pg_pack_tree(int32_t num_nodes, const int32_t* parent, const int32_t* seg_lens,
                       int32_t* position_ids_dev, void* tables_dev, int64_t table_bytes,
                       pg_layout* layout, pg_stream_t stream) {
  int64_t T = 0, bytes = 0;
  pg_status st = pg_pack_tree_size(num_nodes, parent, seg_lens, &T, &bytes);
  if (st != PG_OK) return st;
  if (!position_ids_dev || !tables_dev || !layout || table_bytes < bytes) {
    set_error("pg_pack_tree: NULL buffer or table buffer smaller than %lld bytes",
              (long long)bytes);
    return PG_ERR_INVALID_ARG;
  }
  std::vector<int32_t> pos((size_t)T);
  std::vector<char> tab((size_t)bytes);
  pg_layout host;
  st = pg_pack_tree_host(num_nodes, parent, seg_lens, pos.data(), tab.data(), bytes, &host);
  if (st != PG_OK) return st;
  return upload_layout(pos, tab, position_ids_dev, tables_dev, host, layout,
                       reinterpret_cast<cudaStream_t>(stream));
}

pg_status pg_pack_padded_size(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                              int32_t max_response_len, const int32_t* response_lens,
                              int64_t* total_tokens, int64_t* table_bytes) {
  Plan p;
  Padded pd;
  pg_status st = plan_padded(num_groups, prefix_len, group_size, max_response_len, response_lens,
                             &pd, &p);
  if (st != PG_OK) return st;
  if (total_tokens) *total_tokens = p.T;
  if (table_bytes) *table_bytes = p.bytes;
  return PG_OK;
}

pg_status pg_pack_padded_host(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                              int32_t max_response_len, const int32_t* response_lens,
                              int32_t* position_ids, void* tables, int64_t table_bytes,
                              pg_layout* layout) {
  Plan p;
  Padded pd;
  pg_status st = plan_padded(num_groups, prefix_len, group_size, max_response_len, response_lens,
                             &pd, &p);
  if (st != PG_OK) return st;
  if (!position_ids || !tables || !layout || table_bytes < p.bytes) {
    set_error("pg_pack_padded_host: NULL buffer or table buffer smaller than %lld bytes",
              (long long)p.bytes);
    return PG_ERR_INVALID_ARG;
  }
  memset(tables, 0, (size_t)p.bytes);
  build_tables(num_groups, pd.lp.data(), pd.gs.data(), pd.rs.data(), p, position_ids,
               static_cast<char*>(tables));
  build_pad_list(num_groups, prefix_len, group_size, pd, p, static_cast<char*>(tables));
  fill_layout(num_groups, p, position_ids, tables, layout);
  return PG_OK;
}

pg_status pg_pack_padded(int32_t num_groups, int32_t prefix_len, int32_t group_size,
                         int32_t max_response_len, const int32_t* response_lens,
                         int32_t* position_ids_dev, void* tables_dev, int64_t table_bytes,
                         pg_layout* layout, pg_stream_t stream) {
  int64_t T = 0, bytes = 0;
  pg_status st = pg_pack_padded_size(num_groups, prefix_len, group_size, max_response_len,
                                     response_lens, &T, &bytes);
  if (st != PG_OK) return st;
  if (!position_ids_dev || !tables_dev || !layout || table_bytes < bytes) {
    set_error("pg_pack_padded: NULL buffer or table buffer smaller than %lld bytes",
              (long long)bytes);
    return PG_ERR_INVALID_ARG;
  }
  std::vector<int32_t> pos((size_t)T);
  std::vector<char> tab((size_t)bytes);
  pg_layout host;
  st = pg_pack_padded_host(num_groups, prefix_len, group_size, max_response_len, response_lens,
                           pos.data(), tab.data(), bytes, &host);
  if (st != PG_OK) return st;
  return upload_layout(pos, tab, position_ids_dev, tables_dev, host, layout,
                       reinterpret_cast<cudaStream_t>(stream));
}

pg_status pg_workspace_size(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                            int32_t heads_kv, int32_t head_dim, const pg_opts* opts, int32_t phase,
                            size_t* bytes) {
  if (!bytes || (phase != 0 && phase != 1)) {
    set_error("pg_workspace_size: bytes is NULL or phase not 0/1");
    return PG_ERR_INVALID_ARG;
  }
  pg_status st = check_attn(layout, dtype, heads_q, heads_kv, head_dim, opts, {},
                            "pg_workspace_size");
  if (st != PG_OK) return st;
  bool rope = opts && opts->rope_theta > 0.f;
  const AttnArgs a = make_args(layout, dtype, heads_q, heads_kv, head_dim, opts, nullptr);
  // A forward that keeps its rotated q/k for the backward uses the backward's layout.
  const int ph = (phase == 0 && rope && (a.flags & PG_FLAG_KEEP_ROTATED)) ? 1 : phase;
  *bytes = ws_plan(layout, dtype, heads_q, heads_kv, head_dim, rope, ph, a).total;
  return PG_OK;
}

pg_status pg_grouped_attn_fwd(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                              int32_t heads_kv, int32_t head_dim, const void* q, const void* k,
                              const void* v, void* o, float* lse, const pg_opts* opts,
                              void* workspace, size_t workspace_bytes, pg_stream_t stream) {
  const char* who = "pg_grouped_attn_fwd";
  pg_status st = check_attn(layout, dtype, heads_q, heads_kv, head_dim, opts, {q, k, v, o, lse},
                            who);
  if (st != PG_OK) return st;
  AttnArgs a = make_args(layout, dtype, heads_q, heads_kv, head_dim, opts,
                         reinterpret_cast<cudaStream_t>(stream));
  bool rope = a.theta > 0.f;
  const bool keep = rope && (a.flags & PG_FLAG_KEEP_ROTATED) != 0;
  WsPlan w = ws_plan(layout, dtype, heads_q, heads_kv, head_dim, rope, keep ? 1 : 0, a);
  if (keep && (a.flags & PG_FLAG_RESPONSES_ONLY)) {
    set_error("%s: PG_FLAG_KEEP_ROTATED is for training steps, not with PG_FLAG_RESPONSES_ONLY",
              who);
    return PG_ERR_INVALID_ARG;
  }
  if (w.total > 0 && (!workspace || workspace_bytes < w.total || !aligned16(workspace))) {
    set_error("%s: workspace must be 16-byte aligned and >= %zu bytes", who, w.total);
    return PG_ERR_INVALID_ARG;
  }
  char* ws = static_cast<char*>(workspace);
  const void* qx = q;
  const void* kx = k;
  const bool responses_only = (a.flags & PG_FLAG_RESPONSES_ONLY) != 0;
  if (responses_only && layout->max_depth > 2) {
    set_error("%s: PG_FLAG_RESPONSES_ONLY needs a two-level layout (pg_pack / pg_pack_padded)",
              who);
    return PG_ERR_UNSUPPORTED;
  }
  // Already-rotated q and k (PG_FLAG_PRE_ROTATED) go to the kernels as they are.
  const bool rotate = rope && !(a.flags & PG_FLAG_PRE_ROTATED);
  if (rotate && responses_only) {
    // Every key is rotated; of q only the response rows, the only ones read.
    st = launch_rope(a, k, ws + w.k_rot, heads_kv, q, ws + w.q_rot, heads_q, false, false,
                     nullptr, nullptr, RopeRows::kAllThenResponses);
    if (st != PG_OK) return st;
    qx = ws + w.q_rot;
    kx = ws + w.k_rot;
  } else if (rotate) {
    // Keeping the rotation for the backward also stores the cos/sin table it rotates dK/dQ back
    // with.
    st = launch_rope(a, q, ws + w.q_rot, heads_q, k, ws + w.k_rot, heads_kv, false, false,
                     keep ? reinterpret_cast<float2*>(ws + w.rope_tab) : nullptr, nullptr);
    if (st != PG_OK) return st;
    qx = ws + w.q_rot;
    kx = ws + w.k_rot;
  }
  if (responses_only) {
    if (!(a.flags & PG_FLAG_SIMT) && score_sm100_supported(a))
      st = launch_score_sm100(
          a, qx, kx, v, o, lse,
          w.part_o == SIZE_MAX ? nullptr : reinterpret_cast<float*>(ws + w.part_o),
          w.part_lse == SIZE_MAX ? nullptr : reinterpret_cast<float*>(ws + w.part_lse));
    else
      st = launch_fwd_simt(a, qx, kx, v, o, lse);
  } else if (!(a.flags & PG_FLAG_SIMT) && fwd_sm100_supported(a)) {
    // Keeping the workspace for the backward: also leave it the log2-domain LSE rows.
    float* lse2_out = keep && bwd_sm100_supported(a) ? reinterpret_cast<float*>(ws + w.lse2)
                                                     : nullptr;
    st = launch_fwd_sm100(a, qx, kx, v, o, lse, lse2_out);
  } else {
    st = launch_fwd_simt(a, qx, kx, v, o, lse);
  }
  if (st != PG_OK || layout->n_pad_rows == 0) return st;
  // Padded layout: o = 0 and lse = +inf on the padding rows.
  return launch_pad_fill(a, o, heads_q, nullptr, 0, nullptr, 0, lse);
}

pg_status pg_grouped_attn_bwd(const pg_layout* layout, pg_dtype dtype, int32_t heads_q,
                              int32_t heads_kv, int32_t head_dim, const void* q, const void* k,
                              const void* v, const void* o, const float* lse, const void* dO,
                              void* dq, void* dk, void* dv, const pg_opts* opts, void* workspace,
                              size_t workspace_bytes, pg_stream_t stream) {
  const char* who = "pg_grouped_attn_bwd";
  pg_status st = check_attn(layout, dtype, heads_q, heads_kv, head_dim, opts,
                            {q, k, v, o, lse, dO, dq, dk, dv}, who);
  if (st != PG_OK) return st;
  AttnArgs a = make_args(layout, dtype, heads_q, heads_kv, head_dim, opts,
                         reinterpret_cast<cudaStream_t>(stream));
  if (a.flags & PG_FLAG_RESPONSES_ONLY) {
    set_error("%s: PG_FLAG_RESPONSES_ONLY is a forward-only option", who);
    return PG_ERR_INVALID_ARG;
  }
  bool rope = a.theta > 0.f;
  WsPlan w = ws_plan(layout, dtype, heads_q, heads_kv, head_dim, rope, 1, a);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) {
    set_error("%s: workspace must be 16-byte aligned and >= %zu bytes", who, w.total);
    return PG_ERR_INVALID_ARG;
  }
  char* ws = static_cast<char*>(workspace);
  const void* qx = q;
  const void* kx = k;
  float2* rope_tab = rope ? reinterpret_cast<float2*>(ws + w.rope_tab) : nullptr;
  // PG_FLAG_PRE_ROTATED: q and k come rotated and pg_rope_table wrote the table.
  if (rope && !(a.flags & PG_FLAG_PRE_ROTATED)) {
    // With PG_FLAG_KEEP_ROTATED the forward left the rotated q/k and the table here.
    if (!(a.flags & PG_FLAG_KEEP_ROTATED)) {
      st = launch_rope(a, q, ws + w.q_rot, heads_q, k, ws + w.k_rot, heads_kv, false, false,
                       rope_tab, nullptr);
      if (st != PG_OK) return st;
    }
    qx = ws + w.q_rot;
    kx = ws + w.k_rot;
  }
  float* Dbuf = reinterpret_cast<float*>(ws + w.Dbuf);
  float* lse2 = reinterpret_cast<float*>(ws + w.lse2);
  float* dq_acc = w.dq_acc == SIZE_MAX ? nullptr : reinterpret_cast<float*>(ws + w.dq_acc);
  float* dk_acc = w.dk_acc == SIZE_MAX ? nullptr : reinterpret_cast<float*>(ws + w.dk_acc);
  // With PG_FLAG_KEEP_ROTATED the tensor-core forward already wrote LSE_2.
  const bool prepared = rope && (a.flags & PG_FLAG_KEEP_ROTATED) && !(a.flags & PG_FLAG_SIMT) &&
                        bwd_sm100_supported(a) && fwd_sm100_supported(a);
  st = launch_bwd_preprocess(a, o, dO, lse, Dbuf, lse2, dq_acc, prepared);
  if (st != PG_OK) return st;
  if (!(a.flags & PG_FLAG_SIMT) && bwd_sm100_supported(a)) {
    // dK (inverse-rotated, cast) and dV are written by the key-major kernel itself.  dQ either
    // comes from the query-major kernel (deterministic) or arrives in the fp32 accumulator and is
    // rotated back and cast here.
    st = launch_bwd_sm100(a, qx, kx, v, dO, lse2, Dbuf, dq_acc, dk, dv, rope_tab);
    if (st != PG_OK) return st;
    if (dq_acc == nullptr)
      st = launch_dq_sm100(a, qx, kx, v, dO, lse2, Dbuf, dq, rope_tab);
    else
      st = launch_rope(a, dq_acc, dq, heads_q, nullptr, nullptr, 0, true, true, nullptr,
                       rope_tab);
  } else {
    st = launch_bwd_simt(a, qx, kx, v, o, lse, dO, Dbuf, dq_acc, dk_acc, dv);
    if (st != PG_OK) return st;
    // dQ and dK of the rotated q/k back to the caller's q/k (inverse rotation) and dtype.
    st = launch_rope(a, dq_acc, dq, heads_q, dk_acc, dk, heads_kv, true, true, nullptr, rope_tab);
  }
  if (st != PG_OK || layout->n_pad_rows == 0) return st;
  // Padded layout: the padding rows' gradients are zero (their queries had no weight; no real
  // query sees their keys); write them as exact zeros.
  return launch_pad_fill(a, dq, heads_q, dk, heads_kv, dv, heads_kv, nullptr);
}

pg_status pg_rope_table(const pg_layout* layout, pg_dtype dtype, int32_t heads_q, int32_t heads_kv,
                        int32_t head_dim, const pg_opts* opts, void* workspace,
                        size_t workspace_bytes, const void** table, pg_stream_t stream) {
  const char* who = "pg_rope_table";
  pg_status st = check_attn(layout, dtype, heads_q, heads_kv, head_dim, opts, {workspace}, who);
  if (st != PG_OK) return st;
  if (!table || !opts || !(opts->flags & PG_FLAG_PRE_ROTATED)) {
    set_error("%s: needs opts with PG_FLAG_PRE_ROTATED and rope_theta > 0, and a table pointer",
              who);
    return PG_ERR_INVALID_ARG;
  }
  const AttnArgs a = make_args(layout, dtype, heads_q, heads_kv, head_dim, opts,
                               reinterpret_cast<cudaStream_t>(stream));
  const WsPlan w = ws_plan(layout, dtype, heads_q, heads_kv, head_dim, true, 1, a);
  if (workspace_bytes < w.total) {
    set_error("%s: workspace must be >= %zu bytes (the backward's)", who, w.total);
    return PG_ERR_INVALID_ARG;
  }
  float2* tab = reinterpret_cast<float2*>(static_cast<char*>(workspace) + w.rope_tab);
  // The RoPE pass with no tensors to rotate writes only the table.
  st = launch_rope(a, nullptr, nullptr, 0, nullptr, nullptr, 0, false, false, tab, nullptr);
  if (st != PG_OK) return st;
  *table = tab;
  return PG_OK;
}

pg_status pg_set_profile(pg_profile* profile) {
  g_profile = profile;
  return PG_OK;
}

pg_status pg_device_status(int32_t clear) {
  int32_t code = 0;
  pg_status st = read_kernel_status(clear != 0, &code);
  if (st != PG_OK) return st;
  return static_cast<pg_status>(code);
}

const char* pg_status_string(pg_status s) {
  switch (s) {
    case PG_OK: return "ok";
    case PG_ERR_INVALID_ARG: return "invalid argument";
    case PG_ERR_UNSUPPORTED: return "unsupported";
    case PG_ERR_CUDA: return "CUDA error";
    case PG_ERR_TIMEOUT: return "bounded wait timed out in a kernel";
    case PG_ERR_DEVICE: return "kernel-side check failed";
  }
  return "unknown status";
}

const char* pg_last_error_message(void) { return g_msg; }

}  // extern "C"
