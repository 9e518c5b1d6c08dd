"""GPU parity of the padded-layout adapter (pg_pack_padded) against the CPU oracle.

A packed problem is scattered into the padded layout of the skill page's Step 3 (every response in
a slot of max_response_len tokens, the slot tail filled with arbitrary finite values, including in
dO).  Through that layout the real rows must match the oracle of the unpadded problem (normwise
2e-2 bf16, 1e-5 fp32), and the padding rows must come out exactly o = 0, lse = +inf,
dq = dk = dv = 0.
"""
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


def padded_rows(B, Lp, G, R, rl):
    """Row of the padded buffer holding each packed row, and the padding rows."""
    real, pad = [], []
    for b in range(B):
        base = b * (Lp + G * R)
        real += list(range(base, base + Lp))
        for i in range(G):
            s0 = base + Lp + i * R
            real += list(range(s0, s0 + rl[b * G + i]))
            pad += list(range(s0 + rl[b * G + i], s0 + R))
    return torch.tensor(real), torch.tensor(pad, dtype=torch.int64)


CASES = [
    # (base workload, B, Lp, G, R, response lengths, Hq, Hkv)
    (2, 2, 150, 3, 70, [70, 1, 33, 0, 64, 70], 4, 2),     # bf16 GQA, RoPE, an empty response
    (1, 1, 300, 4, 130, [128, 1, 130, 97], 4, 4),         # bf16 MHA (the 1/sqrt(128) recipe)
    (0, 1, 256, 4, 64, [32, 48, 64, 16], 2, 2),           # the fp32 workload's lengths, padded
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"w{c[0]}")
@pytest.mark.parametrize("path", ["default", "simt"])
def test_padded_layout_matches_unpadded_oracle(case, path):
    wi, B, Lp, G, R, rl, hq, hkv = case
    base = workloads.WORKLOADS[wi]
    w = workloads.small_variant(base, prefix_len=Lp, suffix_lens=rl, heads_q=hq, heads_kv=hkv)
    prob = workloads.make_problem(w, prefix_lens=[Lp] * B, group_sizes=[G] * B, suffix_lens=rl)
    real, pad = padded_rows(B, Lp, G, R, rl)
    Tp = B * (Lp + G * R)
    gen = torch.Generator().manual_seed(7)

    def scatter(x):
        out = torch.randn((Tp,) + tuple(x.shape[1:]), generator=gen).to(x.dtype)  # finite filler
        out[real] = x
        return out

    qp, kp, vp, dop = (scatter(t) for t in (prob.q, prob.k, prob.v, prob.do))
    dev = torch.device("cuda")
    lay = api.pack_padded(B, Lp, G, R, rl, dev)
    assert lay.total_tokens == Tp and lay.struct.n_pad_rows == pad.numel()
    flags = _lib.PG_FLAG_SIMT if path == "simt" else 0
    q, k, v, do = (t.to(dev) for t in (qp, kp, vp, dop))
    o, lse = api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta, flags=flags)
    dq, dk, dv = api.grouped_attn_bwd(lay, q, k, v, o, lse, do, rope_theta=w.rope_theta,
                                      flags=flags)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    got = {n: t.float().cpu() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    if pad.numel():
        for n in ["o", "dq", "dk", "dv"]:
            assert bool((got[n][pad] == 0).all()), n
        assert bool(torch.isposinf(got["lse"][:, pad]).all())
    lay0 = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    ref = orc.repeated_prefix(lay0, prob.q, prob.k, prob.v, prob.do, theta=w.rope_theta)
    errs = {}
    for n in ["o", "dq", "dk", "dv"]:
        errs[n] = orc.normwise_error(got[n][real], getattr(ref, n))
    errs["lse"] = orc.normwise_error(got["lse"][:, real], ref.lse)
    assert all(e <= TOL[w.dtype] for e in errs.values()), errs


def test_padded_responses_only_forward():
    w = workloads.small_variant(workloads.WORKLOADS[4], prefix_len=700, suffix_lens=[3, 1, 4, 2],
                                heads_q=8, heads_kv=2)
    B, Lp, G, R, rl = 1, 700, 4, 5, [3, 1, 4, 2]
    prob = workloads.make_problem(w)
    real, pad = padded_rows(B, Lp, G, R, rl)
    Tp = B * (Lp + G * R)

    def scatter(x):
        out = torch.zeros((Tp,) + tuple(x.shape[1:]), dtype=x.dtype)
        out[real] = x
        return out

    dev = torch.device("cuda")
    lay = api.pack_padded(B, Lp, G, R, rl, dev)
    q, k, v = (scatter(t).to(dev) for t in (prob.q, prob.k, prob.v))
    o = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[1], Tp), float("nan"), device=dev)
    api.grouped_attn_fwd(lay, q, k, v, rope_theta=w.rope_theta,
                         flags=_lib.PG_FLAG_RESPONSES_ONLY, out=o, lse=lse)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    o, lse = o.float().cpu(), lse.cpu()
    assert bool((o[pad] == 0).all()) and bool(torch.isposinf(lse[:, pad]).all())
    lay0 = orc.pack_layout(prob.prefix_lens, prob.group_sizes, prob.suffix_lens)
    rows0 = [t for t in range(lay0.total_tokens) if int(lay0.token_segment[t]) >= 0]
    ref_o, ref_lse = orc.response_rows(lay0, prob.q, prob.k, prob.v, rows0, theta=w.rope_theta)
    rows_p = real[rows0]
    assert orc.normwise_error(o[rows_p], ref_o) <= 2e-2
    assert orc.normwise_error(lse[:, rows_p], ref_lse) <= 2e-2
