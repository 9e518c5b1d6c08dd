"""CPU oracle for Prefix Grouper grouped attention.  TEST INFRASTRUCTURE ONLY.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may import this
module.  The CUDA library and its Python binding never call it, and it calls nothing of theirs: the
two sides share only the seeded input generator (``workloads.py``), which holds no arithmetic of the
method.

What it computes is the plain definition the method claims to reproduce exactly: the
repeated-prefix baseline.  Prefix Grouper (abstract page, "Prefix Grouper: Efficient GRPO Training
through Shared-Prefix Forward") states that encoding [P; R1; ...; RG] once yields the same forward
outputs and backward gradients as encoding every [P; Ri] separately.  The Pith review ("What carries
the argument", "Load-bearing premise") fixes what must match: position IDs exactly as in the
repeated-prefix baseline, and masks such that each suffix token sees the same causal context it has
in the baseline and never another response.  So for every group and every response i this oracle
materialises the sequence [P; Ri], gives it positions 0 .. Lp+ri-1, applies RoPE, runs full causal
softmax attention with an explicit backward, and maps the copies back onto the packed layout:

* suffix rows of O / LSE / dQ / dK / dV come from their own copy;
* prefix rows of O / LSE come from copy 0 (causality makes every copy's prefix rows identical);
* the prefix rows of dQ / dK / dV are the SUM over the G copies -- the Pith review ("major
  comments", Appendix A.1 objection) states that the gradient of the single shared prefix must equal
  the sum of the gradients of the G baseline prefix copies;
* the upstream gradient dO at a prefix row is routed into copy 0 only.  The packed function's VJP is
  unique, so any routing whose weights sum to one gives the same result (a test checks 1/G routing).

A second, independent formulation (``packed_dense``) runs one
attention over the packed sequence with a dense mask built from the baseline's visibility relation.
The two must agree to fp64 rounding.

Everything is float64 and uses plain PyTorch CPU tensor ops (matmul, exp, log, sum).  There is no
tiling, fusion or online softmax: queries are processed in blocks of rows only to bound memory; each
row's softmax is computed from its full row of scores, exactly as written below.

Readings of points the pages leave open (all stated here so a reader can check them by eye):

* softmax scale = d ** -0.5 (the skill page's sketch divides scores by a garbled power of head_dim);
* RoPE is the rotate-half form: for k < d/2 the pair (x[k], x[k + d/2]) is rotated by the angle
  pos * theta ** (-2k/d); theta == 0 disables RoPE.  The pages fix only that positions match the
  baseline;
* GQA: query head h reads key/value head h // (Hq // Hkv);
* no dropout (Pith review, Section 2.2 objection: exact equivalence needs none);
* the skill page's PrefixGroupedAttention sketch (mean-pooled prefix Q/K/V, unmasked softmax) is not
  followed: it contradicts the identical-outputs claim.

Parity unpinned: none.  Every function here is pinned by tests that do not call it alone: the
packing by hand-computed fixtures, RoPE by its complex-number form and group properties, attention by
torch's own scaled_dot_product_attention and autograd (G = 1 and Lp = 0 reduce to that routine),
finite differences, closed forms (Q = 0, constant V) and the packed dense-mask formulation; the
comparison helper normwise_error by hand-worked values (denominator, sign, the skipped non-finite
reference entries, a NaN in the compared tensor, the near-zero branch).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch

F64 = torch.float64


# ------------------------------------------------------------------------------------------------
# Packing and metadata
# ------------------------------------------------------------------------------------------------

@dataclasses.dataclass
class PackedLayout:
    """Integer description of the packed sequence [P_b; R_b1; ...; R_bG] for every group b.

    Sequential concatenation of the prefix and all responses is the skill page's "Sequential
    Concatenation" (Architecture Overview) and the Pith review's [P; R1; ...; RG] ("Core claim").
    Responses are packed back to back without padding.
    """

    prefix_lens: List[int]
    group_sizes: List[int]
    suffix_lens: List[int]
    group_start: torch.Tensor        # int64 [B+1]: first packed row of each group, then T
    segment_start: torch.Tensor      # int64 [S]: first packed row of each response
    position_ids: torch.Tensor       # int64 [T]: the token's position in its baseline [P; Ri]
    token_group: torch.Tensor        # int64 [T]
    token_segment: torch.Tensor      # int64 [T]: response index (group-major), -1 for prefix rows

    @property
    def total_tokens(self) -> int:
        return int(self.group_start[-1])


def pack_layout(prefix_lens: Sequence[int], group_sizes: Sequence[int],
                suffix_lens: Sequence[int]) -> PackedLayout:
    """Offsets and position IDs of the packed layout.

    Position IDs are those of the repeated-prefix baseline (Pith review, "What carries the
    argument"): prefix token j of a group has position j, and token j of response i has position
    Lp + j, restarting for every response, because in the baseline every response follows its own
    copy of the prefix.
    """
    B = len(prefix_lens)
    assert len(group_sizes) == B and sum(group_sizes) == len(suffix_lens)
    assert all(x >= 0 for x in prefix_lens) and all(x >= 0 for x in group_sizes)
    assert all(x >= 0 for x in suffix_lens)
    group_start, segment_start, pos, tg, ts = [], [], [], [], []
    row, seg = 0, 0
    for b in range(B):
        group_start.append(row)
        lp = prefix_lens[b]
        for j in range(lp):
            pos.append(j)
            tg.append(b)
            ts.append(-1)
        row += lp
        for _ in range(group_sizes[b]):
            r = suffix_lens[seg]
            segment_start.append(row)
            for j in range(r):
                pos.append(lp + j)
                tg.append(b)
                ts.append(seg)
            row += r
            seg += 1
    group_start.append(row)
    i64 = lambda xs: torch.tensor(xs, dtype=torch.int64)
    return PackedLayout(list(prefix_lens), list(group_sizes), list(suffix_lens), i64(group_start),
                        i64(segment_start), i64(pos), i64(tg), i64(ts))


def baseline_rows(layout: PackedLayout, b: int, i: Optional[int]) -> torch.Tensor:
    """Packed row indices forming the baseline sequence [P_b; R_bi] (i = None: [P_b] alone)."""
    g0 = int(layout.group_start[b])
    rows = list(range(g0, g0 + layout.prefix_lens[b]))
    if i is not None:
        s0 = int(layout.segment_start[i])
        rows += list(range(s0, s0 + layout.suffix_lens[i]))
    return torch.tensor(rows, dtype=torch.int64)


def group_segments(layout: PackedLayout, b: int) -> List[int]:
    first = sum(layout.group_sizes[:b])
    return list(range(first, first + layout.group_sizes[b]))


def visibility_mask(layout: PackedLayout) -> torch.Tensor:
    """Dense bool [T, T] mask: mask[t, s] is True when packed query t attends to packed key s.

    Built from the baseline only: a query sees exactly the keys that precede it (inclusive) in the
    baseline sequence [P; Ri] its copy lives in (causal attention), mapped back to packed rows.  A
    prefix query sees the prefix keys up to itself; a query of response i sees the whole prefix and
    response i up to itself, never another response (Pith review, "What carries the argument").
    """
    T = layout.total_tokens
    mask = torch.zeros((T, T), dtype=torch.bool)
    for b in range(len(layout.prefix_lens)):
        segs = group_segments(layout, b)
        for i in (segs if segs else [None]):
            rows = baseline_rows(layout, b, i)
            n = rows.numel()
            causal = torch.tril(torch.ones((n, n), dtype=torch.bool))
            mask[rows[:, None], rows[None, :]] |= causal
    return mask


def pair_count_from_mask(layout: PackedLayout) -> int:
    """Visible (query, key) pairs of grouped attention, counted from the mask."""
    return int(visibility_mask(layout).sum())


def repeated_pair_count(layout: PackedLayout) -> int:
    """Visible pairs of the repeated-prefix baseline, counted by materialising every copy."""
    total = 0
    for b in range(len(layout.prefix_lens)):
        segs = group_segments(layout, b)
        for i in (segs if segs else [None]):
            n = baseline_rows(layout, b, i).numel()
            total += int(torch.tril(torch.ones((n, n), dtype=torch.bool)).sum())
    return total


# ------------------------------------------------------------------------------------------------
# RoPE
# ------------------------------------------------------------------------------------------------

def rope_angles(pos: torch.Tensor, d: int, theta: float) -> torch.Tensor:
    """[L, d/2] float64 angles pos * theta ** (-2k/d)."""
    k = torch.arange(d // 2, dtype=F64)
    inv_freq = torch.pow(torch.tensor(float(theta), dtype=F64), -2.0 * k / d)
    return pos.to(F64)[:, None] * inv_freq[None, :]


def rope_rotate(x: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Rotate-half RoPE of x [L, H, d] at positions pos [L]; theta == 0 returns x."""
    if theta == 0:
        return x
    d = x.shape[-1]
    a = rope_angles(pos, d, theta)[:, None, :]
    c, s = torch.cos(a), torch.sin(a)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)


def rope_rotate_vjp(g: torch.Tensor, pos: torch.Tensor, theta: float) -> torch.Tensor:
    """Gradient through rope_rotate: the transpose of a rotation is the rotation by minus the angle."""
    if theta == 0:
        return g
    d = g.shape[-1]
    a = rope_angles(pos, d, theta)[:, None, :]
    c, s = torch.cos(a), torch.sin(a)
    g1, g2 = g[..., : d // 2], g[..., d // 2:]
    return torch.cat([g1 * c + g2 * s, g2 * c - g1 * s], dim=-1)


# ------------------------------------------------------------------------------------------------
# Softmax attention over one sequence with an arbitrary boolean mask, one head
# ------------------------------------------------------------------------------------------------

ROW_BLOCK = 1024


def masked_attention_fwd(q, k, v, mask_fn, scale):
    """O = softmax(scale * q k^T + mask) v and the natural-log LSE, for q [L, d], k, v [N, d].

    mask_fn(r0, r1) returns the bool [r1-r0, N] visibility of rows r0..r1-1.  Every row must see at
    least one key.  Rows are processed in blocks only to bound memory.
    """
    L = q.shape[0]
    O = torch.empty((L, v.shape[1]), dtype=F64)
    lse = torch.empty((L,), dtype=F64)
    for r0 in range(0, L, ROW_BLOCK):
        r1 = min(L, r0 + ROW_BLOCK)
        S = (q[r0:r1] @ k.T) * scale
        S = S.masked_fill(~mask_fn(r0, r1), float("-inf"))
        m = S.max(dim=1, keepdim=True).values
        E = torch.exp(S - m)
        den = E.sum(dim=1, keepdim=True)
        O[r0:r1] = (E / den) @ v
        lse[r0:r1] = (m + torch.log(den))[:, 0]
    return O, lse


def masked_attention_bwd(q, k, v, O, lse, dO, mask_fn, scale):
    """Explicit backward of masked_attention_fwd for the loss sum(dO * O).

    P = exp(scale q k^T - lse) on visible pairs, D = rowsum(dO * O), dP = dO v^T,
    dS = P * (dP - D), dv = P^T dO, dq = scale dS k, dk = scale dS^T q.
    """
    L = q.shape[0]
    dq = torch.empty_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    D = (dO * O).sum(dim=1)
    for r0 in range(0, L, ROW_BLOCK):
        r1 = min(L, r0 + ROW_BLOCK)
        S = (q[r0:r1] @ k.T) * scale
        P = torch.exp(S - lse[r0:r1, None])
        P = P.masked_fill(~mask_fn(r0, r1), 0.0)
        dv += P.T @ dO[r0:r1]
        dP = dO[r0:r1] @ v.T
        dS = P * (dP - D[r0:r1, None])
        dq[r0:r1] = scale * (dS @ k)
        dk += scale * (dS.T @ q[r0:r1])
    return dq, dk, dv


def causal_mask_fn(n_keys):
    def fn(r0, r1):
        return torch.arange(n_keys)[None, :] <= torch.arange(r0, r1)[:, None]
    return fn


# ------------------------------------------------------------------------------------------------
# The repeated-prefix baseline (the oracle proper)
# ------------------------------------------------------------------------------------------------

@dataclasses.dataclass
class AttnResult:
    o: torch.Tensor                  # [T, Hq, d] float64 (NaN on heads not computed)
    lse: torch.Tensor                # [Hq, T] float64
    dq: Optional[torch.Tensor] = None   # [T, Hq, d]
    dk: Optional[torch.Tensor] = None   # [T, Hkv, d] (valid for kv heads whose q heads all ran)
    dv: Optional[torch.Tensor] = None


def _kv_head(h, Hq, Hkv):
    return h // (Hq // Hkv)


def repeated_prefix(layout: PackedLayout, q, k, v, do=None, *, theta: float = 0.0,
                    scale: Optional[float] = None, q_heads: Optional[Sequence[int]] = None,
                    groups: Optional[Sequence[int]] = None, prefix_do_weights=None,
                    check_prefix_copies: bool = True) -> AttnResult:
    """Grouped attention computed as the repeated-prefix baseline (forward, and backward if do).

    q [T, Hq, d], k / v [T, Hkv, d], do [T, Hq, d] in the packed order, any float dtype (upcast to
    float64).  q_heads / groups restrict the work to a subset (heads and groups are independent);
    rows and heads outside the subset are NaN.  prefix_do_weights(G) -> list of G weights summing to
    one routes dO at prefix rows into the copies (default: all into copy 0).
    """
    q, k, v = q.to(F64), k.to(F64), v.to(F64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    assert Hq % Hkv == 0 and T == layout.total_tokens
    scale = d ** -0.5 if scale is None else scale
    q_heads = list(range(Hq)) if q_heads is None else list(q_heads)
    groups = list(range(len(layout.prefix_lens))) if groups is None else list(groups)
    nan = float("nan")
    O = torch.full((T, Hq, d), nan, dtype=F64)
    LSE = torch.full((Hq, T), nan, dtype=F64)
    bwd = do is not None
    if bwd:
        do = do.to(F64)
        dQ = torch.full((T, Hq, d), nan, dtype=F64)
        dK = torch.full((T, Hkv, d), nan, dtype=F64)
        dV = torch.full((T, Hkv, d), nan, dtype=F64)
        kv_heads = sorted({_kv_head(h, Hq, Hkv) for h in q_heads})
    for b in groups:
        g0, g1 = int(layout.group_start[b]), int(layout.group_start[b + 1])
        lp = layout.prefix_lens[b]
        segs = group_segments(layout, b)
        copies = segs if segs else [None]
        G = len(copies)
        w = prefix_do_weights(G) if prefix_do_weights is not None else [1.0] + [0.0] * (G - 1)
        if bwd:
            for kh in kv_heads:
                dK[g0:g1, kh] = 0.0
                dV[g0:g1, kh] = 0.0
            for h in q_heads:
                dQ[g0:g1, h] = 0.0
        for ci, i in enumerate(copies):
            rows = baseline_rows(layout, b, i)
            n = rows.numel()
            if n == 0:
                continue
            pos = torch.arange(n)          # baseline positions 0 .. Lp + ri - 1
            qi = rope_rotate(q[rows], pos, theta)
            ki = rope_rotate(k[rows], pos, theta)
            vi = v[rows]
            mfn = causal_mask_fn(n)
            dki = torch.zeros((n, Hkv, d), dtype=F64)
            dvi = torch.zeros((n, Hkv, d), dtype=F64)
            for h in q_heads:
                kh = _kv_head(h, Hq, Hkv)
                o, lse = masked_attention_fwd(qi[:, h], ki[:, kh], vi[:, kh], mfn, scale)
                if ci == 0:
                    O[rows[:lp], h] = o[:lp]
                    LSE[h, rows[:lp]] = lse[:lp]
                elif check_prefix_copies and lp > 0:
                    err = (o[:lp] - O[rows[:lp], h]).abs().max().item()
                    ref = O[rows[:lp], h].abs().max().item()
                    assert err <= 1e-12 * max(ref, 1.0), "prefix rows differ between copies"
                O[rows[lp:], h] = o[lp:]
                LSE[h, rows[lp:]] = lse[lp:]
                if bwd:
                    doi = do[rows, h].clone()
                    doi[:lp] *= w[ci]
                    dq_r, dk_r, dv_r = masked_attention_bwd(qi[:, h], ki[:, kh], vi[:, kh], o, lse,
                                                            doi, mfn, scale)
                    dQ[rows, h] += rope_rotate_vjp(dq_r[:, None, :], pos, theta)[:, 0]
                    dki[:, kh] += dk_r
                    dvi[:, kh] += dv_r
            if bwd:
                dki = rope_rotate_vjp(dki, pos, theta)
                for kh in kv_heads:
                    dK[rows, kh] += dki[:, kh]
                    dV[rows, kh] += dvi[:, kh]
    if bwd:
        return AttnResult(O, LSE, dQ, dK, dV)
    return AttnResult(O, LSE)


def response_rows(layout: PackedLayout, q, k, v, rows: Sequence[int], *, theta: float = 0.0,
                  scale: Optional[float] = None, q_heads: Optional[Sequence[int]] = None):
    """Forward O and LSE of selected response rows, straight from the baseline's definition.

    Packed row t = token j of response i of group b is row Lp + j of the baseline sequence
    [P_b; R_bi].  Causal attention makes that row depend only on the baseline rows 0 .. Lp + j, so
    it is computed from them alone: positions 0 .. Lp + j, RoPE, scores against those Lp + j + 1
    keys, softmax, weighted sum of the values.  This is the quantity scored when many short
    responses are judged against one long context (Pith review, "Core claim"), and it keeps the
    cost per row at O(Lp d) so rows of very long prefixes can be sampled.
    Returns (O [len(rows), len(q_heads), d], LSE [len(q_heads), len(rows)]) in float64.
    """
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    q_heads = list(range(Hq)) if q_heads is None else list(q_heads)
    O = torch.empty((len(rows), len(q_heads), d), dtype=F64)
    LSE = torch.empty((len(q_heads), len(rows)), dtype=F64)
    prefix_k = {}     # group -> its prefix keys rotated at positions 0 .. Lp-1 (same in every copy)
    for n, t in enumerate(rows):
        i = int(layout.token_segment[t])
        assert i >= 0, "response_rows takes response rows only"
        b = int(layout.token_group[t])
        lp = layout.prefix_lens[b]
        j = t - int(layout.segment_start[i])
        seq = baseline_rows(layout, b, i)[: lp + j + 1]
        pos = torch.arange(seq.numel())
        if b not in prefix_k:
            prefix_k[b] = rope_rotate(k[seq[:lp]].to(F64), pos[:lp], theta)
        kr = torch.cat([prefix_k[b], rope_rotate(k[seq[lp:]].to(F64), pos[lp:], theta)])
        vr = v[seq].to(F64)
        qr = rope_rotate(q[t:t + 1].to(F64), pos[-1:], theta)[0]
        for hn, h in enumerate(q_heads):
            kh = _kv_head(h, Hq, Hkv)
            s_ = (kr[:, kh] @ qr[h]) * scale
            m = s_.max()
            e = torch.exp(s_ - m)
            den = e.sum()
            O[n, hn] = (e / den) @ vr[:, kh]
            LSE[hn, n] = m + torch.log(den)
    return O, LSE


# ------------------------------------------------------------------------------------------------
# Second formulation: one attention over the packed sequence with a dense mask
# ------------------------------------------------------------------------------------------------

def packed_dense(layout: PackedLayout, q, k, v, do=None, *, theta: float = 0.0,
                 scale: Optional[float] = None) -> AttnResult:
    """Grouped attention as one masked attention over the packed sequence (small T only)."""
    q, k, v = q.to(F64), k.to(F64), v.to(F64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    mask = visibility_mask(layout)
    mfn = lambda r0, r1: mask[r0:r1]
    pos = layout.position_ids
    qr = rope_rotate(q, pos, theta)
    kr = rope_rotate(k, pos, theta)
    O = torch.empty((T, Hq, d), dtype=F64)
    LSE = torch.empty((Hq, T), dtype=F64)
    if do is not None:
        do = do.to(F64)
        dQr = torch.empty((T, Hq, d), dtype=F64)
        dKr = torch.zeros((T, Hkv, d), dtype=F64)
        dV = torch.zeros((T, Hkv, d), dtype=F64)
    for h in range(Hq):
        kh = _kv_head(h, Hq, Hkv)
        o, lse = masked_attention_fwd(qr[:, h], kr[:, kh], v[:, kh], mfn, scale)
        O[:, h], LSE[h] = o, lse
        if do is not None:
            dq, dk, dv = masked_attention_bwd(qr[:, h], kr[:, kh], v[:, kh], o, lse, do[:, h], mfn,
                                              scale)
            dQr[:, h] = dq
            dKr[:, kh] += dk
            dV[:, kh] += dv
    if do is None:
        return AttnResult(O, LSE)
    return AttnResult(O, LSE, rope_rotate_vjp(dQr, pos, theta), rope_rotate_vjp(dKr, pos, theta), dV)


# ------------------------------------------------------------------------------------------------
# Nested prefixes (trees): one history replayed against many continuations
# ------------------------------------------------------------------------------------------------
#
# The Pith review ("Reading between the lines") names multi-turn, tree-shaped sharing: one history
# reused by many continuations.  The baseline generalises directly: every root-to-leaf path of
# segments is one sequence of its own (positions 0 .. its length - 1) run through causal attention.
# Packed, the segments follow each other in depth-first preorder; a node's tokens come from the
# first path through it (all paths give the same values by causality), the upstream gradient at a
# token is routed into that first path, and every gradient is summed over all paths.

@dataclasses.dataclass
class TreeLayout:
    parent: List[int]
    lens: List[int]
    start: List[int]
    end: List[int]
    children: List[List[int]]
    position_ids: torch.Tensor       # int64 [T]: position in the token's root-to-leaf sequence
    token_node: torch.Tensor         # int64 [T]

    @property
    def total_tokens(self) -> int:
        return int(self.end[-1]) if self.end else 0


def tree_layout(parent: Sequence[int], lens: Sequence[int]) -> TreeLayout:
    """Rows of the nodes in the listed order, which must be a depth-first preorder."""
    n = len(parent)
    assert len(lens) == n and all(x >= 0 for x in lens)
    children = [[] for _ in range(n)]
    start, end, off, stack, row = [], [], [], [], 0
    for i in range(n):
        p = parent[i]
        assert -1 <= p < i
        while stack and stack[-1] != p:
            stack.pop()
        assert p < 0 or stack, "not a depth-first preorder"
        if p >= 0:
            children[p].append(i)
        off.append(off[p] + lens[p] if p >= 0 else 0)
        start.append(row)
        row += lens[i]
        end.append(row)
        stack.append(i)
    pos, node = [], []
    for i in range(n):
        pos += [off[i] + j for j in range(lens[i])]
        node += [i] * lens[i]
    i64 = lambda xs: torch.tensor(xs, dtype=torch.int64)
    return TreeLayout(list(parent), list(lens), start, end, children, i64(pos), i64(node))


def tree_paths(tl: TreeLayout) -> List[List[int]]:
    """Root-to-leaf node paths, leaves in listed order."""
    paths = []
    for i in range(len(tl.parent)):
        if not tl.children[i]:
            path, a = [], i
            while a >= 0:
                path.append(a)
                a = tl.parent[a]
            paths.append(path[::-1])
    return paths


def tree_visibility(tl: TreeLayout) -> torch.Tensor:
    """bool [T, T]: row t sees key s iff s's node is an ancestor of t's node, or the same node and
    s <= t."""
    T = tl.total_tokens
    n = len(tl.parent)
    anc = torch.zeros((n, n), dtype=torch.bool)      # anc[a, b]: a is b or an ancestor of b
    for b in range(n):
        a = b
        while a >= 0:
            anc[a, b] = True
            a = tl.parent[a]
    nt, ns = tl.token_node[:, None], tl.token_node[None, :]
    t = torch.arange(T)[:, None]
    s = torch.arange(T)[None, :]
    same = nt == ns
    return (anc[ns, nt] & ~same) | (same & (s <= t))


def tree_repeated(tl: TreeLayout, q, k, v, do=None, *, theta: float = 0.0,
                  scale: Optional[float] = None) -> AttnResult:
    """Grouped attention over nested prefixes computed path by path (the baseline)."""
    q, k, v = q.to(F64), k.to(F64), v.to(F64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    nan = float("nan")
    O = torch.full((T, Hq, d), nan, dtype=F64)
    LSE = torch.full((Hq, T), nan, dtype=F64)
    bwd = do is not None
    if bwd:
        do = do.to(F64)
        dQ = torch.zeros((T, Hq, d), dtype=F64)
        dK = torch.zeros((T, Hkv, d), dtype=F64)
        dV = torch.zeros((T, Hkv, d), dtype=F64)
    done = torch.zeros(T, dtype=torch.bool)          # rows already taken from an earlier path
    for path in tree_paths(tl):
        rows = torch.cat([torch.arange(tl.start[a], tl.end[a]) for a in path])
        m = rows.numel()
        if m == 0:
            continue
        pos = torch.arange(m)
        first = ~done[rows]                          # this path is the first one through these rows
        qi, ki, vi = rope_rotate(q[rows], pos, theta), rope_rotate(k[rows], pos, theta), v[rows]
        mfn = causal_mask_fn(m)
        dki = torch.zeros((m, Hkv, d), dtype=F64)
        dvi = torch.zeros((m, Hkv, d), dtype=F64)
        for h in range(Hq):
            kh = _kv_head(h, Hq, Hkv)
            o, lse = masked_attention_fwd(qi[:, h], ki[:, kh], vi[:, kh], mfn, scale)
            O[rows[first], h] = o[first]
            LSE[h, rows[first]] = lse[first]
            if bwd:
                doi = do[rows, h] * first[:, None].to(F64)      # dO routed to the first path
                a_, b_, c_ = masked_attention_bwd(qi[:, h], ki[:, kh], vi[:, kh], o, lse, doi, mfn,
                                                  scale)
                dQ[rows, h] += rope_rotate_vjp(a_[:, None, :], pos, theta)[:, 0]
                dki[:, kh] += b_
                dvi[:, kh] += c_
        if bwd:
            dK[rows] += rope_rotate_vjp(dki, pos, theta)
            dV[rows] += dvi
        done[rows] = True
    if bwd:
        return AttnResult(O, LSE, dQ, dK, dV)
    return AttnResult(O, LSE)


def tree_packed_dense(tl: TreeLayout, q, k, v, do=None, *, theta: float = 0.0,
                      scale: Optional[float] = None) -> AttnResult:
    """Second formulation: one attention over the packed rows with the tree's dense mask."""
    q, k, v = q.to(F64), k.to(F64), v.to(F64)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = d ** -0.5 if scale is None else scale
    mask = tree_visibility(tl)
    mfn = lambda r0, r1: mask[r0:r1]
    pos = tl.position_ids
    qr, kr = rope_rotate(q, pos, theta), rope_rotate(k, pos, theta)
    O = torch.empty((T, Hq, d), dtype=F64)
    LSE = torch.empty((Hq, T), dtype=F64)
    if do is not None:
        do = do.to(F64)
        dQr = torch.empty((T, Hq, d), dtype=F64)
        dKr = torch.zeros((T, Hkv, d), dtype=F64)
        dV = torch.zeros((T, Hkv, d), dtype=F64)
    for h in range(Hq):
        kh = _kv_head(h, Hq, Hkv)
        o, lse = masked_attention_fwd(qr[:, h], kr[:, kh], v[:, kh], mfn, scale)
        O[:, h], LSE[h] = o, lse
        if do is not None:
            a_, b_, c_ = masked_attention_bwd(qr[:, h], kr[:, kh], v[:, kh], o, lse, do[:, h], mfn,
                                              scale)
            dQr[:, h] = a_
            dKr[:, kh] += b_
            dV[:, kh] += c_
    if do is None:
        return AttnResult(O, LSE)
    return AttnResult(O, LSE, rope_rotate_vjp(dQr, pos, theta), rope_rotate_vjp(dKr, pos, theta), dV)


# ------------------------------------------------------------------------------------------------
# Comparison helper used by the tests
# ------------------------------------------------------------------------------------------------

def normwise_error(x: torch.Tensor, ref: torch.Tensor) -> float:
    """max|x - ref| / max|ref| over the finite entries of ref (the tolerance form the tests use).

    A reference that is zero up to rounding (max|ref| < 1e-12, e.g. the key gradient of a
    single-token sequence) is compared absolutely instead.
    """
    x = x.to(F64)
    ok = torch.isfinite(ref)
    if not bool(ok.any()):
        return 0.0
    den = ref[ok].abs().max().item()
    num = (x[ok] - ref[ok]).abs().max().item()
    return num / den if den >= 1e-12 else num
