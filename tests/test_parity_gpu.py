"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Tolerances (normwise: max|x - ref| / max|ref| per tensor, against the fp64 oracle on the same
inputs): 1e-5 for the fp32 path, 2e-2 for bf16, on O, LSE, dQ, dK and dV.  Small cases span several
tiles and ragged tails; the full-size workloads run in the benchmark's launch configuration and are
compared on sampled heads/groups the oracle computes exactly.
"""
import math

import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run_gpu(prob, flags=0, theta=None, keep_rotated=False):
    """Forward + backward through the C ABI; outputs start as NaN so unwritten elements show.
    keep_rotated: the benchmark's call pattern (one backward-sized workspace shared by both calls,
    the forward leaving rotated q / k and the cos/sin table in it)."""
    w = prob.workload
    theta = w.rope_theta if theta is None else theta
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    ws = None
    if keep_rotated:
        flags |= _lib.PG_FLAG_KEEP_ROTATED
        opts = api.make_opts(theta, 0.0, flags)
        ws = api._workspace(api.workspace_size(lay, q.dtype, q.shape[1], k.shape[1], q.shape[2],
                                               opts, 1), dev)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=dev)
    api.grouped_attn_fwd(lay, q, k, v, rope_theta=theta, flags=flags, out=o, lse=lse,
                         workspace=ws)
    dq = torch.full_like(q, float("nan"))
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=theta, flags=flags, dq=dq, dk=dk,
                         dv=dv, workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    out = {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    for n, t in out.items():
        assert bool(torch.isfinite(t).all()), f"{n} has unwritten or non-finite elements"
    return out


def compare(prob, got, tol, q_heads=None, groups=None, theta=None):
    w = prob.workload
    theta = w.rope_theta if theta is None else theta
    lay = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    ref = orc.repeated_prefix(lay, prob.q, prob.k, prob.v, prob.do, theta=theta, q_heads=q_heads,
                              groups=groups)
    errs = {}
    for n in ["o", "lse", "dq", "dk", "dv"]:
        r = getattr(ref, n)
        errs[n] = orc.normwise_error(got[n], r)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"parity failed (tol {tol}): {errs}"
    return errs


SMALL = [
    # (workload index, prefix_lens, group_sizes, suffix_lens, heads_q, heads_kv)
    (0, None, None, None, None, None),                                   # the fp32 workload, full
    (0, [150, 0], [4, 2], [1, 77, 130, 0, 65, 3], 4, 2),                 # fp32, ragged, GQA
    (1, [300], [4], [64, 1, 127, 129], 4, 4),                            # bf16 MHA, RoPE 1e4
    (2, [200, 130], [3, 2], [64, 100, 1, 250, 7], 8, 2),                 # bf16 GQA, two groups
    (3, [520], [5], [256, 1024, 300, 17, 129], 4, 1),                    # bf16 GQA, theta 5e5
]


PATH_FLAGS = {"default": 0, "simt": _lib.PG_FLAG_SIMT, "det": _lib.PG_FLAG_DETERMINISTIC}


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"w{c[0]}")
@pytest.mark.parametrize("path", ["default", "simt", "det"])
def test_small_cases(case, path):
    wi, plens, gsz, rs, hq, hkv = case
    w = workloads.WORKLOADS[wi]
    if plens is not None:
        w = workloads.small_variant(w, prefix_len=plens[0], suffix_lens=rs, heads_q=hq,
                                    heads_kv=hkv)
    prob = workloads.make_problem(w, prefix_lens=plens, group_sizes=gsz, suffix_lens=rs)
    got = run_gpu(prob, flags=PATH_FLAGS[path])
    compare(prob, got, TOL[w.dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("lens", [
    ([0], [3], [5, 1, 9]),          # empty prefix: independent causal responses
    ([9], [0], []),                 # a prefix with no responses
    ([1], [1], [0]),                # a single token
    ([64], [2], [64, 64]),          # exact tile multiples
    ([3, 0, 70], [1, 2, 0], [0, 2, 1]),  # empty pieces everywhere
])
@pytest.mark.parametrize("det", [False, True])
def test_edge_cases(dtype, lens, det):
    plens, gsz, rs = lens
    base = workloads.WORKLOADS[0 if dtype == "f32" else 2]
    w = workloads.small_variant(base, prefix_len=plens[0], suffix_lens=rs, heads_q=4, heads_kv=2)
    w = workloads.dataclasses.replace(w, head_dim=128, rope_theta=100.0)
    prob = workloads.make_problem(w, prefix_lens=plens, group_sizes=gsz, suffix_lens=rs)
    got = run_gpu(prob, flags=_lib.PG_FLAG_DETERMINISTIC if det else 0)
    compare(prob, got, TOL[dtype])


@pytest.mark.parametrize("path", ["default", "det"])
def test_no_cross_response_leakage_on_gpu(path):
    """Perturbing every input of response 1 (q, k, v and the upstream gradient dO) leaves the
    prefix rows and the other responses' rows bit-identical: O, LSE, dK, dV and (on the
    deterministic path, whose dQ has a fixed summation order) dQ.  Only the prefix dK / dV, which
    sum over all responses' queries, may change -- and must, since response 1 sees the prefix."""
    w = workloads.small_variant(workloads.WORKLOADS[1], prefix_len=200, suffix_lens=[90, 140, 33],
                                heads_q=2, heads_kv=2)
    prob = workloads.make_problem(w)
    flags = PATH_FLAGS[path]
    a = run_gpu(prob, flags=flags)
    sl = slice(290, 430)                 # response 1
    prob.q[sl] = -prob.q[sl]
    prob.k[sl] = prob.k[sl] * 2
    prob.v[sl] = prob.v[sl] + 1
    prob.do[sl] = prob.do[sl] * -3
    b = run_gpu(prob, flags=flags)
    compare(prob, b, TOL[w.dtype])
    keep = torch.ones(prob.total_tokens, dtype=torch.bool)
    keep[sl] = False
    resp = keep.clone()
    resp[:200] = False                   # rows of responses 0 and 2
    assert torch.equal(a["o"][keep], b["o"][keep])
    assert torch.equal(a["lse"][:, keep], b["lse"][:, keep])
    assert torch.equal(a["dk"][resp], b["dk"][resp])
    assert torch.equal(a["dv"][resp], b["dv"][resp])
    if path == "det":
        assert torch.equal(a["dq"][keep], b["dq"][keep])
    else:
        assert orc.normwise_error(b["dq"][keep], a["dq"][keep].double()) < 1e-5
    assert not torch.equal(a["o"][sl], b["o"][sl])
    assert not torch.equal(a["dk"][:200], b["dk"][:200])
    assert not torch.equal(a["dv"][:200], b["dv"][:200])


def test_prefix_gradient_is_deterministic():
    w = workloads.small_variant(workloads.WORKLOADS[2], prefix_len=400,
                                suffix_lens=[100, 300, 5, 260], heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    a = run_gpu(prob)
    b = run_gpu(prob)
    assert torch.equal(a["dk"], b["dk"]) and torch.equal(a["dv"], b["dv"])
    assert torch.equal(a["o"], b["o"]) and torch.equal(a["lse"], b["lse"])


def test_deterministic_flag_makes_dq_bitwise_reproducible():
    # With PG_FLAG_DETERMINISTIC every gradient, dq included, is bitwise identical run to run and
    # dk / dv are those of the default path (the same key-major kernel computes them).
    w = workloads.small_variant(workloads.WORKLOADS[2], prefix_len=1000,
                                suffix_lens=[100, 300, 5, 260, 77], heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    det = _lib.PG_FLAG_DETERMINISTIC
    a, b, c = run_gpu(prob, flags=det), run_gpu(prob, flags=det), run_gpu(prob)
    for n in ["dq", "dk", "dv"]:
        assert torch.equal(a[n], b[n]), n
    assert torch.equal(a["dk"], c["dk"]) and torch.equal(a["dv"], c["dv"])
    assert orc.normwise_error(a["dq"].double(), c["dq"].double()) < 1e-2


# ---------------------------------------------------------------- full-size workloads ----------

@pytest.mark.parametrize("wi,q_heads,groups,flags", [
    (1, [0, 31], None, 0),          # bf16 MHA, P=4096, G=8, R=512: two of 32 heads
    (2, [4, 5, 6, 7], [0, 5], 0),   # bf16 GQA, 8 groups: kv head 1, groups 0 and 5
    (1, [7, 20], None, _lib.PG_FLAG_DETERMINISTIC),   # the deterministic backward at full size
])
def test_full_size_sampled(wi, q_heads, groups, flags):
    w = workloads.WORKLOADS[wi]
    prob = workloads.make_problem(w)
    got = run_gpu(prob, flags=flags)
    errs = compare(prob, got, TOL[w.dtype], q_heads=q_heads, groups=groups)
    print(w.name, errs)


def test_full_size_long_prefix():
    """P=16384, G=16 at full size, in the benchmark's launch configuration, compared element by
    element on every row of one query head and its KV head.

    The upstream gradient of query heads 9, 10 and 11 is zeroed, so the GPU's dK / dV of KV head 2
    is the contribution of query head 8 alone (zero dO gives P^T dO = 0 and dS = P * (dO V^T -
    rowsum(dO * O)) = 0).  The oracle runs the repeated-prefix baseline for head 8 over all 16
    copies [P; R_i]: O, LSE and dQ of head 8 and dK, dV of KV head 2 on every packed row, the
    prefix rows of dK / dV being the sum over the 16 copies (reduction depth up to ~26.6k query
    rows per prefix key).  A cheap property is checked as well: summed over keys, dV equals the sum
    of dO over all rows of the KV head's query heads."""
    w = workloads.WORKLOADS[3]
    prob = workloads.make_problem(w)
    prob.do[:, 9:12] = 0
    got = run_gpu(prob, keep_rotated=True)
    lay = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    h, kh = 8, 2
    ref = orc.repeated_prefix(lay, prob.q, prob.k, prob.v, prob.do, theta=w.rope_theta,
                              q_heads=[h], check_prefix_copies=False)
    tol = TOL[w.dtype]
    lp = prob.prefix_lens[0]
    errs = {}
    for n in ["o", "dq"]:
        errs[n] = orc.normwise_error(got[n][:, h], getattr(ref, n)[:, h])
    errs["lse"] = orc.normwise_error(got["lse"][h], ref.lse[h])
    for n in ["dk", "dv"]:
        errs[n] = orc.normwise_error(got[n][:, kh], getattr(ref, n)[:, kh])
        errs[n + "_prefix"] = orc.normwise_error(got[n][:lp, kh], getattr(ref, n)[:lp, kh])
    print(w.name, errs)
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"parity failed (tol {tol}): {errs}"
    rep = w.heads_q // w.heads_kv
    do_sum = prob.do.double().view(prob.total_tokens, w.heads_kv, rep, w.head_dim).sum(dim=(0, 2))
    dv_sum = got["dv"].double().sum(dim=0)
    assert orc.normwise_error(dv_sum, do_sum) <= tol


@pytest.mark.parametrize("path", ["default", "det", "simt", "f32"])
def test_keep_rotated_reuses_the_forward_rotation(path):
    # The forward leaves rotated q/k and the cos/sin table in a backward-sized workspace; the
    # backward then skips its own rotation.  Same kernels on the same rotated values: results are
    # bitwise those of the default call pair, and match the oracle.
    det = path == "det"
    w = workloads.small_variant(workloads.WORKLOADS[0 if path == "f32" else 2], prefix_len=700,
                                suffix_lens=[100, 300, 5, 260], heads_q=8, heads_kv=2)
    w = workloads.dataclasses.replace(w, rope_theta=1e4)
    prob = workloads.make_problem(w)
    base = {"default": 0, "det": _lib.PG_FLAG_DETERMINISTIC, "simt": _lib.PG_FLAG_SIMT,
            "f32": 0}[path]
    ref = run_gpu(prob, flags=base)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    flags = base | _lib.PG_FLAG_KEEP_ROTATED
    opts = api.make_opts(w.rope_theta, 0.0, flags)
    ws = api._workspace(api.workspace_size(lay, q.dtype, w.heads_q, w.heads_kv, w.head_dim,
                                           opts, 1), dev)
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags,
                                  workspace=ws)
    dq, dk, dv = api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=w.rope_theta,
                                      flags=flags, workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    got = {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    # the SIMT and fp32 paths are deterministic too
    for n in ["o", "lse", "dk", "dv"] + (["dq"] if path != "default" else []):
        assert torch.equal(got[n], ref[n]), n
    compare(prob, got, TOL[w.dtype])


@pytest.mark.parametrize("flags", [0, _lib.PG_FLAG_RESPONSES_ONLY])
def test_outputs_only_16_byte_aligned(flags):
    # The API takes 16-byte aligned output and workspace pointers; the kernels write o (and the
    # scoring kernel its split partials in the workspace) with 32-byte stores only where the
    # buffer is 32-byte aligned.  Buffers 16 bytes off a 32-byte boundary get the same values.
    w = workloads.small_variant(workloads.WORKLOADS[3], prefix_len=1100, suffix_lens=[70, 1, 129],
                                heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    q, k, v = (t.to(dev) for t in (prob.q, prob.k, prob.v))
    n_ws = api.workspace_size(lay, q.dtype, q.shape[1], k.shape[1], q.shape[2],
                              api.make_opts(w.rope_theta, 0.0, flags), 0)
    outs = []
    for shift in (0, 8):                       # elements of bf16: 0 and 16 bytes
        big = torch.full((q.numel() + 16,), float("nan"), dtype=q.dtype, device=dev)
        ws_big = torch.empty(n_ws + 64, dtype=torch.uint8, device=dev)
        assert big.data_ptr() % 32 == 0 and ws_big.data_ptr() % 32 == 0
        o = big[shift:shift + q.numel()].view(q.shape)
        ws = ws_big[2 * shift:2 * shift + n_ws]
        lse = torch.full((q.shape[1], q.shape[0]), float("nan"), device=dev)
        api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags, out=o, lse=lse,
                             workspace=ws)
        torch.cuda.synchronize()
        assert api.device_status() == 0
        outs.append((o.float().cpu(), lse.cpu()))
    assert torch.equal(outs[0][0].nan_to_num(), outs[1][0].nan_to_num())
    assert torch.equal(outs[0][1].nan_to_num(), outs[1][1].nan_to_num())
    rows = slice(1100, None) if flags else slice(None)
    assert bool(torch.isfinite(outs[1][0][rows]).all())


@pytest.mark.parametrize("path", ["default", "det"])
def test_many_work_items_all_rows(path):
    # More forward work items (query-tile pairs x heads) and backward key blocks than the GPU has
    # SMs, at a size the oracle checks on every row: the forward's CTAs claim pending items
    # (cluster launch control) and run several each, with items of different lengths (groups of
    # three prefix lengths), so every row of o / lse and of the gradients comes from a claimed item
    # as often as from a launched one.
    plens = [130, 260, 40] * 14
    gsz = [2, 1, 3] * 14
    rs = [30, 1, 99, 7, 12, 64] * 14
    w = workloads.small_variant(workloads.WORKLOADS[2], prefix_len=plens[0], suffix_lens=rs,
                                heads_q=8, heads_kv=2, num_groups=len(plens))
    prob = workloads.make_problem(w, prefix_lens=plens, group_sizes=gsz, suffix_lens=rs)
    dev_lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, torch.device("cuda"))
    assert dev_lay.struct.n_tiles[4] * w.heads_q > 2 * 152          # 256-row forward items
    got = run_gpu(prob, flags=PATH_FLAGS[path])
    compare(prob, got, TOL[w.dtype])
