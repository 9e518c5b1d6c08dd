"""GPU parity of the pre-rotated path: RoPE applied in the q / k projection's GEMM epilogue
(pg_gemm_bf16_rope, cos/sin table from pg_rope_table) and attention calls with
PG_FLAG_PRE_ROTATED.

* the table against the oracle's fp64 angles (cos and sin within 1e-6);
* the RoPE GEMM against a plain fp64 GEMM of the same bf16 operands rotated by the oracle's fp64
  RoPE (normwise <= 4e-3: one bf16 rounding of the output), for head_dim 128 and 64, ragged row
  counts and a partial last column tile;
* the attention forward and backward on q, k rotated beforehand (by the oracle, rounded to bf16)
  against the oracle on the un-rotated inputs (normwise 2e-2, as every bf16 parity test): the
  gradients must still be those with respect to the un-rotated q and k;
* the responses-only forward on pre-rotated q, k.
The decoder layer with the fused projections is covered by test_layer_gpu.py.
"""
import pytest
import torch

from oracle import prefix_grouper_oracle as orc
from shared_prefix_grouped_gb300 import _lib, api, workloads
from shared_prefix_grouped_gb300.build import build

pytestmark = pytest.mark.gpu

PRE = _lib.PG_FLAG_PRE_ROTATED
BF = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()


def table_for(lay, Hq, Hkv, d, theta, flags):
    ws = api._workspace(api.workspace_size(lay, BF, Hq, Hkv, d, api.make_opts(theta, 0.0, flags),
                                           1), torch.device("cuda"))
    return ws, api.rope_table(lay, BF, Hq, Hkv, d, ws, rope_theta=theta, flags=flags)


GEMM_CASES = [
    # (head_dim, N, prefix_lens, group_sizes, suffix_lens) -> M = total tokens
    (128, 384, [200], [2], [60, 40]),                 # M = 300; second column tile half full
    (64, 512, [64, 0], [1, 2], [1, 30, 34]),          # M = 129; four heads per column tile
    (128, 4096, [700], [3], [100, 150, 50]),          # M = 1000; the q-projection width
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: f"d{c[0]}_n{c[1]}")
def test_gemm_rope_matches_rotated_fp64_gemm(case):
    d, N, plens, gsz, rs = case
    theta, K = 5e5, 256
    dev = torch.device("cuda")
    lay = api.pack(plens, gsz, rs, dev)
    M = lay.total_tokens
    g = torch.Generator().manual_seed(11)
    a = torch.randn(M, K, generator=g).to(BF)
    b = (torch.randn(N, K, generator=g) * K ** -0.5).to(BF)
    ws, tab = table_for(lay, N // d, 1, d, theta, PRE)
    c = api.gemm_bf16_rope(a.to(dev), b.to(dev), tab, M, d)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    pos = lay.position_ids.cpu()
    # the table sits at the start of the workspace: float2 [M][d/2]
    t = ws[: M * (d // 2) * 8].view(torch.float32).view(M, d // 2, 2).cpu().double()
    ang = orc.rope_angles(pos, d, theta)
    assert (t[..., 0] - torch.cos(ang)).abs().max() <= 1e-6
    assert (t[..., 1] - torch.sin(ang)).abs().max() <= 1e-6
    ref = orc.rope_rotate((a.double() @ b.double().T).view(M, N // d, d), pos, theta).view(M, N)
    assert orc.normwise_error(c.float().cpu(), ref) <= 4e-3


ATTN_FLAGS = [0, _lib.PG_FLAG_KEEP_ROTATED, _lib.PG_FLAG_DETERMINISTIC,
              _lib.PG_FLAG_KEEP_ROTATED | _lib.PG_FLAG_DETERMINISTIC, _lib.PG_FLAG_SIMT]


@pytest.mark.parametrize("flags", ATTN_FLAGS, ids=lambda f: f"flags{f}")
def test_pre_rotated_attention_matches_oracle(flags):
    w = workloads.small_variant(workloads.WORKLOADS[2], prefix_len=300, suffix_lens=[100, 5, 130],
                                heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    pos = lay.position_ids.cpu()
    theta = w.rope_theta
    qr = orc.rope_rotate(prob.q.double(), pos, theta).to(BF)
    kr = orc.rope_rotate(prob.k.double(), pos, theta).to(BF)
    f = PRE | flags
    ws, _ = table_for(lay, w.heads_q, w.heads_kv, w.head_dim, theta, f)
    q, k, v, do = (t.to(dev) for t in (qr, kr, prob.v, prob.do))
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=theta, flags=f, workspace=ws)
    dq, dk, dv = api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=theta, flags=f,
                                      workspace=ws)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    ref = orc.repeated_prefix(orc.pack_layout(prob.prefix_lens, prob.group_sizes,
                                              prob.suffix_lens),
                              prob.q, prob.k, prob.v, prob.do, theta=theta)
    got = dict(o=o, dq=dq, dk=dk, dv=dv)
    errs = {n: orc.normwise_error(t.float().cpu(), getattr(ref, n)) for n, t in got.items()}
    errs["lse"] = orc.normwise_error(lse.cpu(), ref.lse)
    assert all(e <= 2e-2 for e in errs.values()), errs


def test_pre_rotated_responses_only_forward():
    w = workloads.small_variant(workloads.WORKLOADS[4], prefix_len=700, suffix_lens=[3, 1, 4, 2],
                                heads_q=8, heads_kv=2)
    prob = workloads.make_problem(w)
    dev = torch.device("cuda")
    lay = api.pack(prob.prefix_lens, prob.group_sizes, prob.suffix_lens, dev)
    pos = lay.position_ids.cpu()
    theta = w.rope_theta
    qr = orc.rope_rotate(prob.q.double(), pos, theta).to(BF).to(dev)
    kr = orc.rope_rotate(prob.k.double(), pos, theta).to(BF).to(dev)
    f = PRE | _lib.PG_FLAG_RESPONSES_ONLY
    o = torch.full_like(qr, float("nan"))
    lse = torch.full((w.heads_q, lay.total_tokens), float("nan"), device=dev)
    api.grouped_attn_fwd(lay, qr, kr, prob.v.to(dev), rope_theta=theta, flags=f, out=o, lse=lse)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    lay0 = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    rows = [t for t in range(lay0.total_tokens) if int(lay0.token_segment[t]) >= 0]
    ref_o, ref_lse = orc.response_rows(lay0, prob.q, prob.k, prob.v, rows, theta=theta)
    assert orc.normwise_error(o.float().cpu()[rows], ref_o) <= 2e-2
    assert orc.normwise_error(lse.cpu()[:, rows], ref_lse) <= 2e-2
