"""Pins for the CPU oracle, checked against things other than the oracle itself.

* the packing: a hand-derived fixture (tests/golden/pack_two_groups.json) and the pair closed forms;
* RoPE: its complex-number form, norm preservation, relative-position invariance, inverse = VJP;
* attention: torch's scaled_dot_product_attention + autograd (G = 1 and Lp = 0 reduce to it),
  central finite differences, closed forms (Q = 0, constant V);
* the method's own claims: repeated-prefix == packed dense-mask formulation (outputs and the summed
  prefix gradient), dO routing independence, no cross-response leakage.
"""
import json
import math
import os

import pytest
import torch
import torch.nn.functional as F

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import flops

F64 = torch.float64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64)


def problem(prefix_lens, group_sizes, suffix_lens, Hq, Hkv, d, seed=0):
    lay = orc.pack_layout(prefix_lens, group_sizes, suffix_lens)
    T = lay.total_tokens
    return (lay, rand((T, Hq, d), seed), rand((T, Hkv, d), seed + 1), rand((T, Hkv, d), seed + 2),
            rand((T, Hq, d), seed + 3))


# ---------------------------------------------------------------- packing -----------------------

def test_pack_matches_hand_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "pack_two_groups.json")))
    lay = orc.pack_layout(fx["prefix_lens"], fx["group_sizes"], fx["suffix_lens"])
    assert lay.total_tokens == fx["total_tokens"]
    assert lay.group_start.tolist() == fx["group_start"]
    assert lay.segment_start.tolist() == fx["segment_start"]
    assert lay.position_ids.tolist() == fx["position_ids"]
    mask = orc.visibility_mask(lay)
    got = [torch.nonzero(mask[t]).flatten().tolist() for t in range(lay.total_tokens)]
    assert got == fx["visible_keys"]
    assert orc.pair_count_from_mask(lay) == fx["grouped_pairs"]
    assert orc.repeated_pair_count(lay) == fx["repeated_pairs"]


@pytest.mark.parametrize("lp,rs", [(0, [3, 1]), (5, []), (7, [0, 4, 9]), (16, [1, 2, 3, 5, 8])])
def test_pair_counts_match_closed_form(lp, rs):
    lay = orc.pack_layout([lp], [len(rs)], rs)
    assert orc.pair_count_from_mask(lay) == flops.group_pairs(lp, rs)
    assert orc.repeated_pair_count(lay) == flops.group_repeated_pairs(lp, rs)


def test_flop_ratio_tends_to_one_over_g():
    # Lemma 2.2 (Pith review, "Core claim"): the cost ratio approaches 1/G when Lp >> |R|.
    G, r = 8, 64
    prev = 1.0
    for lp in [64, 1024, 16384, 1 << 20, 1 << 26]:
        ratio = flops.group_pairs(lp, [r] * G) / flops.group_repeated_pairs(lp, [r] * G)
        assert ratio < prev
        prev = ratio
    assert abs(prev - 1.0 / G) < 1e-5


# ---------------------------------------------------------------- RoPE --------------------------

def test_rope_matches_complex_rotation():
    d, L, theta = 16, 11, 100.0
    x = rand((L, 3, d), 7)
    pos = torch.arange(L) * 3 + 1
    got = orc.rope_rotate(x, pos, theta)
    z = torch.complex(x[..., : d // 2], x[..., d // 2:])
    freq = theta ** (-(torch.arange(0, d, 2, dtype=F64)) / d)
    rot = torch.polar(torch.ones(L, d // 2, dtype=F64), pos[:, None].to(F64) * freq[None, :])
    zr = z * rot[:, None, :]
    assert torch.allclose(got, torch.cat([zr.real, zr.imag], dim=-1), atol=1e-13, rtol=0)


def test_rope_properties():
    d, theta = 8, 50.0
    q, k = rand((1, 1, d), 1), rand((1, 1, d), 2)
    # position 0 is the identity; rotations preserve norms; scores depend on m - n only
    assert torch.equal(orc.rope_rotate(q, torch.tensor([0]), theta), q)
    qr = orc.rope_rotate(q, torch.tensor([37]), theta)
    assert abs(qr.norm().item() - q.norm().item()) < 1e-12
    def score(m, n):
        return (orc.rope_rotate(q, torch.tensor([m]), theta) * orc.rope_rotate(k, torch.tensor([n]), theta)).sum().item()
    assert abs(score(9, 4) - score(105, 100)) < 1e-11
    assert abs(score(9, 4) - score(4, 9)) > 1e-6
    # the VJP of a rotation is its inverse
    x = rand((5, 2, d), 3)
    pos = torch.arange(5) + 3
    assert torch.allclose(orc.rope_rotate_vjp(orc.rope_rotate(x, pos, theta), pos, theta), x, atol=1e-13)


# ---------------------------------------------------------------- attention vs library ----------

def sdpa_reference(q, k, v, do, causal_mask=None):
    """torch SDPA (library routine) on [L, H, d] tensors with autograd; returns O, dq, dk, dv."""
    q, k, v = (t.detach().clone().requires_grad_(True) for t in (q, k, v))
    Hq, Hkv = q.shape[1], k.shape[1]
    rep = Hq // Hkv
    kk = k.repeat_interleave(rep, dim=1)
    vv = v.repeat_interleave(rep, dim=1)
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None], kk.transpose(0, 1)[None],
                                       vv.transpose(0, 1)[None], is_causal=True)[0].transpose(0, 1)
    (o * do).sum().backward()
    return o.detach(), q.grad, k.grad, v.grad


@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (4, 2)])
def test_single_response_is_textbook_causal_attention(Hq, Hkv):
    lay, q, k, v, do = problem([13], [1], [6], Hq, Hkv, 8, seed=11)
    res = orc.repeated_prefix(lay, q, k, v, do)
    o, dq, dk, dv = sdpa_reference(q, k, v, do)
    for a, b in [(res.o, o), (res.dq, dq), (res.dk, dk), (res.dv, dv)]:
        assert orc.normwise_error(a, b) < 1e-12


def rope_complex_diff(x, pos, theta):
    """Differentiable complex-form RoPE written independently of the oracle."""
    d = x.shape[-1]
    freq = theta ** (-(torch.arange(0, d, 2, dtype=F64)) / d)
    a = pos[:, None].to(F64) * freq[None, :]
    c, s = torch.cos(a)[:, None], torch.sin(a)[:, None]
    re, im = x[..., : d // 2], x[..., d // 2:]
    return torch.cat([re * c - im * s, re * s + im * c], dim=-1)


def test_single_response_with_rope_matches_autograd():
    theta = 30.0
    lay, q, k, v, do = problem([9], [1], [5], 2, 1, 8, seed=21)
    res = orc.repeated_prefix(lay, q, k, v, do, theta=theta)
    pos = torch.arange(14)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = F.scaled_dot_product_attention(
        rope_complex_diff(qq, pos, theta).transpose(0, 1)[None],
        rope_complex_diff(kk, pos, theta).repeat_interleave(2, dim=1).transpose(0, 1)[None],
        vv.repeat_interleave(2, dim=1).transpose(0, 1)[None], is_causal=True)[0].transpose(0, 1)
    (o * do).sum().backward()
    for a, b in [(res.o, o.detach()), (res.dq, qq.grad), (res.dk, kk.grad), (res.dv, vv.grad)]:
        assert orc.normwise_error(a, b) < 1e-12


def test_empty_prefix_is_independent_causal_attention():
    rs = [4, 1, 0, 7]
    lay, q, k, v, do = problem([0], [4], rs, 2, 2, 8, seed=31)
    res = orc.repeated_prefix(lay, q, k, v, do)
    s = 0
    for r in rs:
        if r:
            sl = slice(s, s + r)
            o, dq, dk, dv = sdpa_reference(q[sl], k[sl], v[sl], do[sl])
            for a, b in [(res.o[sl], o), (res.dq[sl], dq), (res.dk[sl], dk), (res.dv[sl], dv)]:
                assert orc.normwise_error(a, b) < 1e-12
        s += r


def test_lse_matches_logsumexp():
    lay, q, k, v, _ = problem([6], [2], [3, 2], 2, 2, 4, seed=41)
    res = orc.repeated_prefix(lay, q, k, v)
    mask = orc.visibility_mask(lay)
    for h in range(2):
        S = (q[:, h] @ k[:, h].T) * 0.5
        S = S.masked_fill(~mask, float("-inf"))
        assert torch.allclose(res.lse[h], torch.logsumexp(S, dim=1), atol=1e-13, rtol=0)


# ---------------------------------------------------------------- finite differences ------------

def test_finite_differences_tiny():
    theta = 10.0
    lay, q, k, v, do = problem([3, 2], [2, 3], [2, 1, 1, 0, 2], 2, 1, 4, seed=51)
    res = orc.repeated_prefix(lay, q, k, v, do, theta=theta)

    def loss(q_, k_, v_):
        return (orc.repeated_prefix(lay, q_, k_, v_, theta=theta).o * do).sum().item()

    h = 1e-6
    for name, x, grad in [("q", q, res.dq), ("k", k, res.dk), ("v", v, res.dv)]:
        fd = torch.empty_like(x)
        for idx in range(x.numel()):
            xp, xm = x.clone(), x.clone()
            xp.view(-1)[idx] += h
            xm.view(-1)[idx] -= h
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd.view(-1)[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert orc.normwise_error(grad, fd) < 1e-7, name


# ---------------------------------------------------------------- closed forms ------------------

def test_zero_queries_average_visible_values():
    lay, _, k, v, do = problem([5, 3], [2, 1], [3, 2, 4], 2, 2, 4, seed=61)
    q = torch.zeros((lay.total_tokens, 2, 4), dtype=F64)
    res = orc.repeated_prefix(lay, q, k, v, do)
    mask = orc.visibility_mask(lay).to(F64)
    cnt = mask.sum(dim=1)
    for h in range(2):
        assert torch.allclose(res.o[:, h], (mask @ v[:, h]) / cnt[:, None], atol=1e-13)
        assert torch.allclose(res.lse[h], torch.log(cnt), atol=1e-13)
    # with q = 0 every score is 0 whatever k is, so dK vanishes
    assert res.dk.abs().max().item() < 1e-13


def test_constant_values_give_constant_output_and_no_qk_gradient():
    lay, q, k, _, do = problem([4], [3], [2, 5, 1], 2, 1, 4, seed=71)
    v = torch.full((lay.total_tokens, 1, 4), 0.75, dtype=F64)
    res = orc.repeated_prefix(lay, q, k, v, do, theta=7.0)
    assert torch.allclose(res.o, torch.full_like(res.o, 0.75), atol=1e-14)
    assert res.dq.abs().max().item() < 1e-13 and res.dk.abs().max().item() < 1e-13
    # sum over keys of dV equals the sum of dO over all query rows (softmax rows sum to one)
    assert torch.allclose(res.dv.sum(dim=(0, 1)), do.sum(dim=(0, 1)), atol=1e-12)


# ---------------------------------------------------------------- the method's claims -----------

CASES = [
    ([7], [3], [2, 5, 1], 2, 2, 8, 0.0),
    ([9, 4], [2, 3], [3, 1, 2, 0, 6], 4, 2, 8, 25.0),
    ([0, 6], [2, 1], [3, 2, 4], 2, 1, 4, 5.0),
    ([5], [0], [], 2, 1, 4, 9.0),
]


@pytest.mark.parametrize("case", CASES)
def test_repeated_prefix_equals_packed_dense(case):
    plens, gsz, rs, Hq, Hkv, d, theta = case
    lay, q, k, v, do = problem(plens, gsz, rs, Hq, Hkv, d, seed=81)
    a = orc.repeated_prefix(lay, q, k, v, do, theta=theta)
    b = orc.packed_dense(lay, q, k, v, do, theta=theta)
    for x, y in [(a.o, b.o), (a.lse, b.lse), (a.dq, b.dq), (a.dk, b.dk), (a.dv, b.dv)]:
        assert orc.normwise_error(x, y) < 1e-12


def test_prefix_do_routing_does_not_matter():
    lay, q, k, v, do = problem([6], [3], [2, 3, 1], 2, 1, 4, seed=91)
    a = orc.repeated_prefix(lay, q, k, v, do, theta=3.0)
    b = orc.repeated_prefix(lay, q, k, v, do, theta=3.0, prefix_do_weights=lambda G: [1.0 / G] * G)
    for x, y in [(a.dq, b.dq), (a.dk, b.dk), (a.dv, b.dv)]:
        assert orc.normwise_error(x, y) < 1e-12


def test_prefix_gradient_is_sum_over_copies():
    # Pith review (Appendix A.1 objection): the shared prefix's gradient equals the sum of the
    # gradients of its G baseline copies.  Check against copies computed one by one.
    lp, rs = 5, [3, 2, 4]
    lay, q, k, v, do = problem([lp], [3], rs, 2, 2, 4, seed=101)
    res = orc.repeated_prefix(lay, q, k, v, do)
    dk_sum = torch.zeros((lp, 2, 4), dtype=F64)
    for i in range(3):
        rows = orc.baseline_rows(lay, 0, i)
        do_i = do[rows].clone()
        if i > 0:
            do_i[:lp] = 0
        _, _, dk, _ = sdpa_reference(q[rows], k[rows], v[rows], do_i)
        dk_sum += dk[:lp]
    assert orc.normwise_error(res.dk[:lp], dk_sum) < 1e-12


def test_no_cross_response_leakage():
    lay, q, k, v, do = problem([6], [3], [3, 4, 2], 2, 1, 4, seed=111)
    a = orc.repeated_prefix(lay, q, k, v, theta=4.0)
    # perturb response 1 (rows 9..12) in q, k and v
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    sl = slice(9, 13)
    q2[sl] += 1.0
    k2[sl] -= 2.0
    v2[sl] *= 3.0
    b = orc.repeated_prefix(lay, q2, k2, v2, theta=4.0)
    keep = [t for t in range(lay.total_tokens) if not (9 <= t < 13)]
    assert torch.equal(a.o[keep], b.o[keep])
    assert torch.equal(a.lse[:, keep], b.lse[:, keep])
    assert not torch.equal(a.o[sl], b.o[sl])


def test_continuing_positions_change_outputs():
    # Negative control for the position-ID reading: positions that continue across responses
    # (instead of restarting at |P|) give different outputs.
    lay, q, k, v, _ = problem([4], [2], [3, 3], 2, 2, 8, seed=121)
    res = orc.repeated_prefix(lay, q, k, v, theta=10.0)
    cont = orc.rope_rotate(q, torch.arange(lay.total_tokens), 10.0)
    kc = orc.rope_rotate(k, torch.arange(lay.total_tokens), 10.0)
    mask = orc.visibility_mask(lay)
    h = 0
    S = (cont[:, h] @ kc[:, h].T) / math.sqrt(8)
    o = torch.softmax(S.masked_fill(~mask, float("-inf")), dim=1) @ v[:, h]
    assert (o[7:] - res.o[7:, h]).abs().max().item() > 1e-3


# ---------------------------------------------------------------- responses-only rows -----------

@pytest.mark.parametrize("case", CASES[:3])
def test_response_rows_match_repeated_prefix(case):
    plens, gsz, rs, Hq, Hkv, d, theta = case
    lay, q, k, v, _ = problem(plens, gsz, rs, Hq, Hkv, d, seed=131)
    full = orc.repeated_prefix(lay, q, k, v, theta=theta)
    rows = [t for t in range(lay.total_tokens) if int(lay.token_segment[t]) >= 0]
    o, lse = orc.response_rows(lay, q, k, v, rows, theta=theta)
    assert orc.normwise_error(o, full.o[rows]) < 1e-12
    assert orc.normwise_error(lse, full.lse[:, rows]) < 1e-12


def test_response_rows_single_response_is_textbook_causal_attention():
    # G = 1 with RoPE: row Lp + j of causal SDPA over [P; R] (rotated by the complex form).
    theta, lp, r = 40.0, 11, 5
    lay, q, k, v, _ = problem([lp], [1], [r], 4, 2, 8, seed=141)
    pos = torch.arange(lp + r)
    o_ref = F.scaled_dot_product_attention(
        rope_complex_diff(q, pos, theta).transpose(0, 1)[None],
        rope_complex_diff(k, pos, theta).repeat_interleave(2, dim=1).transpose(0, 1)[None],
        v.repeat_interleave(2, dim=1).transpose(0, 1)[None], is_causal=True)[0].transpose(0, 1)
    rows = list(range(lp, lp + r))
    o, _ = orc.response_rows(lay, q, k, v, rows, theta=theta, q_heads=[1, 3])
    assert orc.normwise_error(o, o_ref[rows][:, [1, 3]]) < 1e-12


# ---------------------------------------------------------------- nested prefixes (trees) ------

TREES = [
    # (parent, lens): depth-first preorder
    ([-1, 0, 1, 1, 0, 4, 4, 4], [5, 3, 2, 4, 2, 1, 3, 2]),        # depth 3, two turns
    ([-1, 0, 1, 2, 2, 0, -1, 6, 6], [4, 2, 3, 1, 2, 3, 3, 2, 0]),  # depth 4, two roots, empty leaf
    ([-1, 0, 0, 2, 2, 2], [0, 3, 2, 2, 1, 3]),                     # empty root
]


def tree_problem(parent, lens, Hq, Hkv, d, seed):
    tl = orc.tree_layout(parent, lens)
    T = tl.total_tokens
    return (tl, rand((T, Hq, d), seed), rand((T, Hkv, d), seed + 1), rand((T, Hkv, d), seed + 2),
            rand((T, Hq, d), seed + 3))


def test_two_level_tree_is_the_grouped_layout():
    # A root with leaf children is exactly [P; R1; ...; RG]: same mask, positions and results.
    lp, rs = 6, [3, 1, 4]
    tl, q, k, v, do = tree_problem([-1, 0, 0, 0], [lp] + rs, 4, 2, 8, seed=151)
    lay = orc.pack_layout([lp], [3], rs)
    assert torch.equal(orc.tree_visibility(tl), orc.visibility_mask(lay))
    assert torch.equal(tl.position_ids, lay.position_ids)
    a = orc.tree_repeated(tl, q, k, v, do, theta=7.0)
    b = orc.repeated_prefix(lay, q, k, v, do, theta=7.0)
    for x, y in [(a.o, b.o), (a.lse, b.lse), (a.dq, b.dq), (a.dk, b.dk), (a.dv, b.dv)]:
        assert orc.normwise_error(x, y) < 1e-12


def test_chain_tree_is_one_causal_sequence():
    # Each node the single child of the previous: one sequence, causal SDPA (complex-form RoPE).
    theta = 20.0
    tl, q, k, v, do = tree_problem([-1, 0, 1, 2], [3, 2, 4, 1], 2, 1, 8, seed=161)
    pos = torch.arange(10)
    assert torch.equal(tl.position_ids, pos)
    res = orc.tree_repeated(tl, q, k, v, do, theta=theta)
    qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = F.scaled_dot_product_attention(
        rope_complex_diff(qq, pos, theta).transpose(0, 1)[None],
        rope_complex_diff(kk, pos, theta).repeat_interleave(2, dim=1).transpose(0, 1)[None],
        vv.repeat_interleave(2, dim=1).transpose(0, 1)[None], is_causal=True)[0].transpose(0, 1)
    (o * do).sum().backward()
    for a, b in [(res.o, o.detach()), (res.dq, qq.grad), (res.dk, kk.grad), (res.dv, vv.grad)]:
        assert orc.normwise_error(a, b) < 1e-12


@pytest.mark.parametrize("tree", TREES)
def test_tree_paths_equal_tree_dense_mask(tree):
    parent, lens = tree
    tl, q, k, v, do = tree_problem(parent, lens, 4, 2, 8, seed=171)
    a = orc.tree_repeated(tl, q, k, v, do, theta=11.0)
    b = orc.tree_packed_dense(tl, q, k, v, do, theta=11.0)
    for x, y in [(a.o, b.o), (a.lse, b.lse), (a.dq, b.dq), (a.dk, b.dk), (a.dv, b.dv)]:
        assert orc.normwise_error(x, y) < 1e-12


def test_tree_shared_turn_gradient_is_sum_over_paths():
    # The gradient of a segment shared by several continuations is the sum over the paths, with
    # the upstream gradient of every row counted once (in the first path through it).
    parent, lens = TREES[0]
    tl, q, k, v, do = tree_problem(parent, lens, 2, 2, 4, seed=181)
    res = orc.tree_repeated(tl, q, k, v, do)
    T = tl.total_tokens
    dk_sum = torch.zeros((T, 2, 4), dtype=F64)
    dv_sum = torch.zeros((T, 2, 4), dtype=F64)
    seen = torch.zeros(T, dtype=torch.bool)
    for path in orc.tree_paths(tl):
        prow = torch.cat([torch.arange(tl.start[a], tl.end[a]) for a in path])
        do_p = do[prow] * (~seen[prow]).to(F64)[:, None, None]
        _, _, dk, dv = sdpa_reference(q[prow], k[prow], v[prow], do_p)
        dk_sum[prow] += dk
        dv_sum[prow] += dv
        seen[prow] = True
    assert orc.normwise_error(res.dk, dk_sum) < 1e-12
    assert orc.normwise_error(res.dv, dv_sum) < 1e-12


def test_tree_no_leakage_between_branches():
    parent, lens = TREES[0]
    tl, q, k, v, _ = tree_problem(parent, lens, 2, 1, 4, seed=191)
    a = orc.tree_repeated(tl, q, k, v, theta=3.0)
    sl = slice(tl.start[1], tl.end[3])                 # turn 1 and its two continuations
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[sl] += 1.0
    k2[sl] -= 2.0
    v2[sl] *= 3.0
    b = orc.tree_repeated(tl, q2, k2, v2, theta=3.0)
    keep = [t for t in range(tl.total_tokens) if not (sl.start <= t < sl.stop)]
    assert torch.equal(a.o[keep], b.o[keep]) and torch.equal(a.lse[:, keep], b.lse[:, keep])
    assert not torch.equal(a.o[sl], b.o[sl])


def test_tree_layout_matches_hand_fixture():
    fx = json.load(open(os.path.join(GOLDEN, "pack_tree_small.json")))
    tl = orc.tree_layout(fx["parent"], fx["seg_lens"])
    assert tl.total_tokens == fx["total_tokens"]
    assert tl.position_ids.tolist() == fx["position_ids"]
    mask = orc.tree_visibility(tl)
    assert [mask[t].nonzero().flatten().tolist() for t in range(tl.total_tokens)] == \
        fx["visible_keys"]
    assert int(mask.sum()) == fx["grouped_pairs"]
    assert orc.tree_paths(tl) == fx["paths"]
    lens = fx["seg_lens"]
    assert sum(n * (n + 1) // 2 for n in (sum(lens[a] for a in p) for p in fx["paths"])) == \
        fx["repeated_pairs"]


# ------------------------------------------------------------------ the comparison helper ------

def test_normwise_error_hand_computed_values():
    """normwise_error = max|x - ref| / max|ref| over the finite entries of ref, values worked by
    hand: a wrong denominator (max|x|, a mean, an elementwise ratio), a dropped abs() or a NaN
    swallowed by the max would each change one of these."""
    nan, inf = float("nan"), float("inf")
    ref = torch.tensor([[1.0, -4.0], [2.0, 0.5]], dtype=F64)
    assert orc.normwise_error(ref.clone(), ref) == 0.0
    x = ref.clone()
    x[0, 1] = -3.0                        # |diff| 1, max|ref| 4
    assert orc.normwise_error(x, ref) == 0.25
    x = ref.clone()
    x[1, 1] = 0.25                        # |diff| 0.25 on the smallest entry: 0.25 / 4
    assert orc.normwise_error(x, ref) == 0.0625
    x = ref.clone()
    x[0, 0] = 9.0                         # |diff| 8; max|x| = 9 must not be the denominator
    assert orc.normwise_error(x, ref) == 2.0
    x = ref.clone()
    x[1, 0] = -2.0                        # sign error: |diff| 4
    assert orc.normwise_error(x, ref) == 1.0
    # x in a narrower dtype is upcast, not compared in its own precision
    assert orc.normwise_error(ref.float(), ref) == 0.0
    assert orc.normwise_error(torch.tensor([1.5], dtype=torch.bfloat16),
                              torch.tensor([2.0], dtype=F64)) == 0.25


def test_normwise_error_non_finite_entries():
    nan, inf = float("nan"), float("inf")
    ref = torch.tensor([1.0, -4.0, 2.0], dtype=F64)
    # a NaN or inf in x where ref is finite must fail any tolerance
    for bad in (nan, inf, -inf):
        x = ref.clone()
        x[2] = bad
        e = orc.normwise_error(x, ref)
        assert not e <= 1e30, (bad, e)
    # entries where ref is not finite (heads or groups the oracle did not compute) are skipped,
    # also for the denominator
    ref2 = torch.tensor([1.0, nan, -2.0, inf], dtype=F64)
    x = torch.tensor([1.5, 123.0, -2.0, -7.0], dtype=F64)
    assert orc.normwise_error(x, ref2) == 0.25
    assert orc.normwise_error(x, torch.full((4,), nan, dtype=F64)) == 0.0


def test_normwise_error_zero_reference_is_absolute():
    # A reference that is zero up to rounding (max|ref| < 1e-12) is compared absolutely.
    ref = torch.tensor([0.0, 5e-13, -1e-13], dtype=F64)
    x = torch.tensor([3e-13, -2e-3, 0.0], dtype=F64)
    assert math.isclose(orc.normwise_error(x, ref), 2e-3 + 5e-13, rel_tol=1e-12)
    # at and above the threshold the error is relative again
    ref = torch.tensor([1e-12, 0.0], dtype=F64)
    x = torch.tensor([2e-12, 0.0], dtype=F64)
    assert math.isclose(orc.normwise_error(x, ref), 1.0, rel_tol=1e-12)
