"""GPU parity for nested prefixes (pg_pack_tree) against the CPU oracle's path-by-path baseline.

Trees of depth 3 to 8 with ragged segments, an empty root and an empty leaf, several roots, GQA and
RoPE; the default (tensor-core, TMA reduce-add dQ), deterministic (query-major dQ) and fp32-SIMT
paths.  Tolerances as for the flat layouts: normwise 2e-2 (bf16), 1e-5 (fp32).
"""
import dataclasses

import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}
FLAGS = {"default": 0, "det": _lib.PG_FLAG_DETERMINISTIC, "simt": _lib.PG_FLAG_SIMT}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run_tree(prob, flags):
    w = prob.workload
    dev = torch.device("cuda")
    lay = api.pack_tree(w.parent, w.lens, dev)
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags)
    dq, dk, dv = api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=w.rope_theta,
                                      flags=flags)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    return {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}


def check(prob, got, tol):
    w = prob.workload
    tl = orc.tree_layout(list(w.parent), list(w.lens))
    ref = orc.tree_repeated(tl, prob.q, prob.k, prob.v, prob.do, theta=w.rope_theta)
    errs = {n: orc.normwise_error(got[n], getattr(ref, n)) for n in ["o", "lse", "dq", "dk", "dv"]}
    assert all(e <= tol for e in errs.values()), errs
    return errs


TREES = [
    # (parent, lens, Hq, Hkv, dtype)
    (*workloads.multi_turn(700, 3, 130, 3, 90), 8, 2, "bf16"),          # context / turns / answers
    ((-1, 0, 1, 2, 2, 0, -1, 6, 6), (129, 64, 300, 7, 70, 5, 80, 40, 0), 4, 4, "bf16"),
    ((-1, 0, 0, 2, 2, 2), (0, 33, 100, 64, 1, 250), 4, 1, "bf16"),
    ((-1, 0, 1, 2, 3, 4, 5, 6), (70, 3, 66, 1, 128, 9, 64, 300), 2, 2, "bf16"),   # depth 8
    ((-1, 0, 1, 1, 0, 4, 4, 4), (96, 40, 20, 33, 17, 1, 60, 25), 2, 2, "f32"),
    # 32 query heads: more forward items than SMs, so the forward's CTAs claim items
    (*workloads.multi_turn(700, 3, 130, 3, 90), 32, 8, "bf16"),
]


@pytest.mark.parametrize("tree", TREES, ids=lambda t: f"n{len(t[0])}_h{t[2]}_{t[4]}")
@pytest.mark.parametrize("path", ["default", "det", "simt"])
def test_tree_matches_path_baseline(tree, path):
    parent, lens, hq, hkv, dtype = tree
    d = 64 if dtype == "f32" else 128
    w = workloads.TreeWorkload("tree_case", dtype, tuple(parent), tuple(lens), hq, hkv, d,
                               rope_theta=1e4, seed=2000 + len(parent))
    prob = workloads.make_tree_problem(w)
    if dtype == "bf16":
        # keep softmax inputs in a moderate range, as the flat bf16 cases
        prob = dataclasses.replace(prob, q=(prob.q.float() * 0.5).to(prob.q.dtype))
    got = run_tree(prob, FLAGS[path])
    check(prob, got, TOL[dtype])


def test_tree_gradients_are_deterministic():
    parent, lens = workloads.multi_turn(500, 2, 200, 3, 120)
    w = workloads.TreeWorkload("tree_det", "bf16", parent, lens, 8, 2, 128, rope_theta=1e4)
    prob = workloads.make_tree_problem(w)
    det = _lib.PG_FLAG_DETERMINISTIC
    a, b = run_tree(prob, det), run_tree(prob, det)
    for n in ["o", "lse", "dq", "dk", "dv"]:
        assert torch.equal(a[n], b[n]), n


def test_tree_workload_sampled():
    # The multi-turn benchmark shape scaled to a size the oracle finishes quickly: 1024-token
    # context, 4 turns of 128, 4 answers of 64 each; every head.
    w = workloads.TREE_WORKLOADS[0]
    parent, lens = workloads.multi_turn(1024, 4, 128, 4, 64)
    w = dataclasses.replace(w, parent=parent, lens=lens, heads_q=8, heads_kv=2)
    prob = workloads.make_tree_problem(w)
    got = run_tree(prob, 0)
    check(prob, got, TOL["bf16"])


def test_tree_keep_rotated_deterministic():
    # A nested layout through the training-step options: one workspace, deterministic backward.
    parent, lens = workloads.multi_turn(600, 3, 150, 2, 100)
    w = workloads.TreeWorkload("tree_keep", "bf16", parent, lens, 8, 2, 128, rope_theta=1e4)
    prob = workloads.make_tree_problem(w)
    dev = torch.device("cuda")
    lay = api.pack_tree(w.parent, w.lens, dev)
    flags = _lib.PG_FLAG_DETERMINISTIC | _lib.PG_FLAG_KEEP_ROTATED
    q, k, v, do = (t.to(dev) for t in (prob.q, prob.k, prob.v, prob.do))
    ws = api._workspace(api.workspace_size(lay, q.dtype, 8, 2, 128,
                                           api.make_opts(w.rope_theta, 0.0, flags), 1), dev)
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags,
                                  workspace=ws)
    dq, dk, dv = api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=w.rope_theta,
                                      flags=flags, workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    got = {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    check(prob, got, TOL["bf16"])
