"""GPU parity of the decoder layer (GEMMs, RMSNorm, SwiGLU, grouped attention through the C ABI).

* a small layer (head_dim 128, hidden 256) against the fp64 CPU layer oracle (repeated-prefix
  baseline), outputs, input gradient and every parameter gradient, normwise <= 2e-2, with RoPE
  applied in the q / k projections' GEMM epilogue (the default) and by the attention call;
* the layer at the full workload's dimensions (hidden 4096, 32/8 heads, head_dim 128, MLP 14336,
  RoPE 5e5) on a short ragged batch (two groups, T = 862) against the same oracle, so every GEMM
  runs at its full K and N;
* the full decoder-layer workload (hidden 4096, 32/8 heads, MLP 14336, B=2, P=8192, G=8, R=1024)
  against the same GPU kernels run on the materialised repeated-prefix layout (every [P; Ri] as
  its own sequence), which the pages say must give identical outputs and parameter gradients.
"""
import pytest
import torch

from oracle import layer_oracle as lo
from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import api, layer, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def run_layer(prob, prefix_lens, group_sizes, suffix_lens, x, dy, fused_rope=True):
    w = prob.workload
    dev = torch.device("cuda")
    lay = api.pack(prefix_lens, group_sizes, suffix_lens, dev)
    W = [t.to(dev) for t in (prob.w_qkv, prob.w_o, prob.w_gu, prob.w_d, prob.g1, prob.g2)]
    kw = dict(heads_q=w.heads_q, heads_kv=w.heads_kv, head_dim=w.head_dim, rope_theta=w.rope_theta,
              eps=w.rms_eps)
    x, dy = x.to(dev), dy.to(dev)
    y, saved = layer.layer_fwd(lay, x, *W, fused_rope=fused_rope, **kw)
    g = layer.layer_bwd(lay, x, *W, saved, dy, **kw)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    return y, g


@pytest.mark.parametrize("fused_rope", [True, False], ids=["rope_in_gemm", "rope_in_attn"])
def test_small_layer_matches_oracle(fused_rope):
    w = workloads.small_layer()
    prob = workloads.make_layer_problem(w, suffix_lens=[70, 1, 129, 64, 30, 200])
    y, g = run_layer(prob, prob.prefix_lens, prob.group_sizes, prob.suffix_lens, prob.x, prob.dy,
                     fused_rope)
    W = (prob.w_qkv, prob.w_o, prob.w_gu, prob.w_d, prob.g1, prob.g2)
    ref = lo.layer_repeated(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, prob.x, prob.dy,
                            W, heads_q=w.heads_q, heads_kv=w.heads_kv, head_dim=w.head_dim,
                            theta=w.rope_theta, eps=w.rms_eps)
    got = dict(y=y, dx=g.dx, w_qkv=g.w_qkv, w_o=g.w_o, w_gu=g.w_gu, w_d=g.w_d, g1=g.g1, g2=g.g2)
    errs = {n: orc.normwise_error(t.float().cpu(), getattr(ref, n)) for n, t in got.items()}
    assert all(e <= TOL for e in errs.values()), errs


def test_full_dims_layer_matches_oracle():
    w = workloads.dataclasses.replace(workloads.LayerWorkload(), name="llama_layer_full_dims_short",
                                      prefix_len=200, group_size=3, num_groups=2)
    prob = workloads.make_layer_problem(w, suffix_lens=[40, 1, 130, 64, 77, 150])
    y, g = run_layer(prob, prob.prefix_lens, prob.group_sizes, prob.suffix_lens, prob.x, prob.dy)
    W = (prob.w_qkv, prob.w_o, prob.w_gu, prob.w_d, prob.g1, prob.g2)
    ref = lo.layer_repeated(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, prob.x, prob.dy,
                            W, heads_q=w.heads_q, heads_kv=w.heads_kv, head_dim=w.head_dim,
                            theta=w.rope_theta, eps=w.rms_eps)
    got = dict(y=y, dx=g.dx, w_qkv=g.w_qkv, w_o=g.w_o, w_gu=g.w_gu, w_d=g.w_d, g1=g.g1, g2=g.g2)
    errs = {n: orc.normwise_error(t.float().cpu(), getattr(ref, n)) for n, t in got.items()}
    print(errs)
    assert all(e <= TOL for e in errs.values()), errs


def repeated_layout(prob):
    """Rows of the materialised [P; Ri] copies and their layout (one group per copy)."""
    lps, gss, rss, idx = [], [], [], []
    s, g0 = 0, 0
    for lp, G in zip(prob.prefix_lens, prob.group_sizes):
        seg0 = g0 + lp
        for i in range(G):
            r = prob.suffix_lens[s + i]
            lps.append(lp)
            gss.append(1)
            rss.append(r)
            idx.append(torch.arange(g0, g0 + lp))
            idx.append(torch.arange(seg0, seg0 + r))
            seg0 += r
        g0 = seg0
        s += G
    return lps, gss, rss, idx


def test_full_layer_grouped_equals_repeated_on_gpu():
    w = workloads.LayerWorkload()
    prob = workloads.make_layer_problem(w)
    y, g = run_layer(prob, prob.prefix_lens, prob.group_sizes, prob.suffix_lens, prob.x, prob.dy)
    lps, gss, rss, idx = repeated_layout(prob)
    rows = torch.cat(idx)
    # upstream gradient of a prefix row goes into the group's first copy only
    dy_rep = prob.dy[rows].clone()
    off, first = 0, True
    k = 0
    for b, (lp, G) in enumerate(zip(prob.prefix_lens, prob.group_sizes)):
        for i in range(G):
            n = lp + rss[k]
            if i > 0:
                dy_rep[off:off + lp] = 0
            off += n
            k += 1
    yr, gr = run_layer(prob, lps, gss, rss, prob.x[rows], dy_rep)
    T = prob.total_tokens
    # outputs: every packed row equals its copy's row (prefix rows from the first copy)
    y_rep = torch.empty_like(y)
    dx_rep = torch.zeros((T, w.hidden), dtype=torch.float32, device=y.device)
    rows_d = rows.to(y.device)
    y_rep[rows_d] = yr  # later copies overwrite prefix rows with identical values
    dx_rep.index_add_(0, rows_d, gr.dx.float())
    assert orc.normwise_error(y.float().cpu(), y_rep.float().cpu().double()) <= TOL
    assert orc.normwise_error(g.dx.float().cpu(), dx_rep.cpu().double()) <= TOL
    for n in ["w_qkv", "w_o", "w_gu", "w_d", "g1", "g2"]:
        e = orc.normwise_error(getattr(g, n).cpu(), getattr(gr, n).cpu().double())
        assert e <= TOL, (n, e)
