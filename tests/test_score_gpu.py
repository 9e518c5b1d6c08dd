"""GPU parity of the responses-only forward (PG_FLAG_RESPONSES_ONLY) against the CPU oracle.

The response rows' O and LSE must match the repeated-prefix baseline (normwise, 2e-2 for bf16 and
1e-5 for fp32); the prefix rows of o and lse must be left exactly as they were (the call does not
write them).  Cases cover the key-split path with its LSE merge, several row blocks per group,
groups of different prefix lengths (one empty prefix, one group without responses), head ratios
that do and do not divide 256, and the full-size scoring workload in the benchmark's launch
configuration, sampled on every key/value head.
"""
import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
RESP = _lib.PG_FLAG_RESPONSES_ONLY


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run_score(prob, flags):
    w = prob.workload
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v = (t.to(dev) for t in (prob.q, prob.k, prob.v))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=dev)
    api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=RESP | flags, out=o, lse=lse)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    return o.float().cpu(), lse.cpu()


def response_row_ids(prob):
    lay = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    return lay, [t for t in range(lay.total_tokens) if int(lay.token_segment[t]) >= 0]


def check(prob, o, lse, tol, q_heads=None):
    lay, rows = response_row_ids(prob)
    w = prob.workload
    heads = list(range(w.heads_q)) if q_heads is None else list(q_heads)
    prefix = [t for t in range(lay.total_tokens) if int(lay.token_segment[t]) < 0]
    # prefix rows untouched, response rows written
    assert bool(torch.isnan(o[prefix]).all()) and bool(torch.isnan(lse[:, prefix]).all())
    assert bool(torch.isfinite(o[rows]).all()) and bool(torch.isfinite(lse[:, rows]).all())
    ref_o, ref_lse = orc.response_rows(lay, prob.q, prob.k, prob.v, rows, theta=w.rope_theta,
                                       q_heads=heads)
    eo = orc.normwise_error(o[rows][:, heads], ref_o)
    el = orc.normwise_error(lse[heads][:, rows], ref_lse)
    assert eo <= tol and el <= tol, (eo, el)
    return eo, el


CASES = [
    # (base workload, prefix_lens, group_sizes, suffix_lens, Hq, Hkv)
    (4, [700], [6], [1, 3, 2, 4, 1, 2], 8, 2),                   # GQA 4:1, one row block, 5 splits
    (1, [300], [4], [64, 1, 127, 129], 4, 4),                    # MHA: 256-token row blocks, 2 blocks
    (4, [500, 0, 64], [3, 2, 0], [2, 5, 1, 3, 4], 8, 2),         # empty prefix, group w/o responses
    (4, [400], [3], [30, 50, 20], 6, 2),                         # 3 heads per kv head: 85-token blocks
    (4, [260], [5], [3, 4, 5, 6, 2], 32, 1),                     # 32 heads per kv head: 8-token blocks
    (3, [1100, 333], [2, 3], [40, 200, 7, 90, 1], 8, 4),         # two groups, longer responses
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"h{c[4]}x{c[5]}_p{c[1][0]}")
@pytest.mark.parametrize("path", ["default", "simt"])
def test_responses_only_small(case, path):
    wi, plens, gsz, rs, hq, hkv = case
    base = workloads.WORKLOADS[wi]
    w = workloads.small_variant(base, prefix_len=plens[0], suffix_lens=rs, heads_q=hq,
                                heads_kv=hkv)
    prob = workloads.make_problem(w, prefix_lens=plens, group_sizes=gsz, suffix_lens=rs)
    o, lse = run_score(prob, _lib.PG_FLAG_SIMT if path == "simt" else 0)
    check(prob, o, lse, TOL[w.dtype])


def test_responses_only_fp32_workload():
    prob = workloads.make_problem(workloads.WORKLOADS[0])
    o, lse = run_score(prob, 0)
    check(prob, o, lse, TOL["f32"])


def test_responses_only_matches_full_forward_rows():
    # The same response rows from the full forward (a different kernel) agree within bf16 rounding.
    w = workloads.small_variant(workloads.WORKLOADS[4], prefix_len=900, suffix_lens=[3, 1, 4, 1, 5],
                                heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    o, lse = run_score(prob, 0)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    of, lf = api.grouped_attn_fwd(lay, prob.q.to(dev), prob.k.to(dev), prob.v.to(dev),
                                  rope_theta=w.rope_theta)
    _, rows = response_row_ids(prob)
    assert orc.normwise_error(o[rows], of.float().cpu()[rows].double()) < 1e-2
    assert orc.normwise_error(lse[:, rows], lf.cpu()[:, rows].double()) < 1e-3


def test_responses_only_is_deterministic_and_leak_free():
    w = workloads.small_variant(workloads.WORKLOADS[4], prefix_len=1500,
                                suffix_lens=[4, 2, 3, 1, 4, 2], heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    o1, l1 = run_score(prob, 0)
    o2, l2 = run_score(prob, 0)
    assert torch.equal(o1.nan_to_num(), o2.nan_to_num()) and torch.equal(l1.nan_to_num(),
                                                                         l2.nan_to_num())
    # perturb response 2 (rows 1506..1508): every other response row is bit-identical
    lo = 1500 + 4 + 2
    sl = slice(lo, lo + 3)
    q2, k2, v2 = prob.q.clone(), prob.k.clone(), prob.v.clone()
    q2[sl] = (q2[sl].float() + 1).to(q2.dtype)
    k2[sl] = (k2[sl].float() - 2).to(k2.dtype)
    v2[sl] = (v2[sl].float() * 3).to(v2.dtype)
    prob2 = workloads.Problem(w, prob.prefix_lens, prob.group_sizes, prob.suffix_lens, q2, k2, v2,
                              prob.do)
    o3, l3 = run_score(prob2, 0)
    _, rows = response_row_ids(prob)
    keep = [t for t in rows if not (lo <= t < lo + 3)]
    assert torch.equal(o1[keep], o3[keep]) and torch.equal(l1[:, keep], l3[:, keep])
    assert not torch.equal(o1[sl], o3[sl])


def test_responses_only_full_size_workload_sampled():
    # The scoring workload at full size, through the same call the benchmark times; every
    # response row checked on two query heads of each key/value head.
    w = workloads.WORKLOADS[4]
    prob = workloads.make_problem(w)
    o, lse = run_score(prob, 0)
    heads = [h for kh in range(w.heads_kv) for h in (4 * kh, 4 * kh + 3)]
    check(prob, o, lse, TOL["bf16"], q_heads=heads)


def test_backward_rejects_responses_only():
    w = workloads.small_variant(workloads.WORKLOADS[4], prefix_len=64, suffix_lens=[2, 3],
                                heads_q=2, heads_kv=1)
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    o, lse = api.grouped_attn_fwd(lay, q, k, v)
    with pytest.raises(_lib.PgError) as e:
        api.grouped_attn_bwd(lay, q, k, v, o, lse, do, flags=RESP)
    assert e.value.status == _lib.PG_ERR_INVALID_ARG
