"""One Llama-style decoder layer over packed shared-prefix groups, composed from the library's
C-ABI kernels (tensor-core GEMMs, RMSNorm, SwiGLU, grouped attention).  Torch only allocates.

Every linear projection and MLP runs over the packed tokens, so a group's shared prefix passes
through them once instead of once per response (abstract page of Prefix Grouper: the shared
prefix is encoded only once; Pith review, "Core claim": the cost tends to 1/G of the baseline).

Forward:  h1 = rmsnorm(x) g1;  q, k, v = h1 W_q^T, h1 W_k^T, h1 W_v^T (RoPE of q and k applied in
          their GEMMs' epilogue, or with fused_rope=False by the attention call);  o = attn(q, k, v);
          x2 = x + o W_o^T;  h2 = rmsnorm(x2) g2;  [g | u] = h2 W_gu^T;  y = x2 + (silu(g) u) W_d^T
Backward: the chain rule through the same steps, weight gradients in fp32.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib, api


@dataclasses.dataclass
class LayerGrads:
    dx: torch.Tensor
    w_qkv: torch.Tensor
    w_o: torch.Tensor
    w_gu: torch.Tensor
    w_d: torch.Tensor
    g1: torch.Tensor
    g2: torch.Tensor


def _views(w_qkv, Hq, Hkv, d):
    nq, nk = Hq * d, Hkv * d
    return w_qkv[:nq], w_qkv[nq:nq + nk], w_qkv[nq + nk:]


def layer_fwd(layout: api.Layout, x, w_qkv, w_o, w_gu, w_d, g1, g2, *, heads_q, heads_kv,
              head_dim, rope_theta, eps, fused_rope: bool = True):
    T, H = x.shape
    Hq, Hkv, d = heads_q, heads_kv, head_dim
    wq, wk, wv = _views(w_qkv, Hq, Hkv, d)
    bf = torch.bfloat16
    h1, _, r1 = api.rmsnorm_fwd(x, g1, eps)
    # One attention workspace for the step: the forward leaves its log2-domain LSE (and, unless
    # the projections rotate q and k themselves, the rotated q/k and the cos/sin table) there for
    # the backward (PG_FLAG_KEEP_ROTATED).
    fused = fused_rope and rope_theta > 0
    flags = _lib.PG_FLAG_KEEP_ROTATED | (_lib.PG_FLAG_PRE_ROTATED if fused else 0)
    ws = api._workspace(api.workspace_size(layout, bf, Hq, Hkv, d,
                                           api.make_opts(rope_theta, 0.0, flags), 1), x.device)
    if fused:
        # RoPE in the q and k projections' epilogue, from the workspace's cos/sin table (which the
        # backward also rotates dq and dk back with).
        tab = api.rope_table(layout, bf, Hq, Hkv, d, ws, rope_theta=rope_theta, flags=flags)
        q = api.gemm_bf16_rope(h1, wq, tab, T, d)
        k = api.gemm_bf16_rope(h1, wk, tab, T, d)
    else:
        q = api.gemm_bf16(h1, wq, out_dtype=bf)
        k = api.gemm_bf16(h1, wk, out_dtype=bf)
    v = api.gemm_bf16(h1, wv, out_dtype=bf)
    o, lse = api.grouped_attn_fwd(layout, q.view(T, Hq, d), k.view(T, Hkv, d), v.view(T, Hkv, d),
                                  rope_theta=rope_theta, flags=flags, workspace=ws)
    a = api.gemm_bf16(o.view(T, Hq * d), w_o, out_dtype=bf)
    h2, x2, r2 = api.rmsnorm_fwd(x, g2, eps, residual=a)
    gu = api.gemm_bf16(h2, w_gu, out_dtype=bf)
    act = api.swiglu_fwd(gu)
    y = x2.clone()
    api.gemm_bf16(act, w_d, out=y, accumulate=True)
    saved = dict(h1=h1, r1=r1, q=q, k=k, v=v, o=o, lse=lse, x2=x2, h2=h2, r2=r2, gu=gu, act=act,
                 attn_ws=ws, attn_flags=flags)
    return y, saved


def layer_bwd(layout: api.Layout, x, w_qkv, w_o, w_gu, w_d, g1, g2, saved, dy, *, heads_q,
              heads_kv, head_dim, rope_theta, eps) -> LayerGrads:
    T, H = x.shape
    Hq, Hkv, d = heads_q, heads_kv, head_dim
    wq, wk, wv = _views(w_qkv, Hq, Hkv, d)
    bf, f32 = torch.bfloat16, torch.float32
    s = saved
    d_act = api.gemm_bf16(dy, w_d, b_mn=True, out_dtype=bf)
    dw_d = api.gemm_bf16(dy, s["act"], a_mn=True, b_mn=True, out_dtype=f32)
    d_gu = api.swiglu_bwd(s["gu"], d_act)
    dh2 = api.gemm_bf16(d_gu, w_gu, b_mn=True, out_dtype=f32)
    dw_gu = api.gemm_bf16(d_gu, s["h2"], a_mn=True, b_mn=True, out_dtype=f32)
    dx2, dg2 = api.rmsnorm_bwd(s["x2"], g2, s["r2"], dh2, dres=dy, dx_dtype=bf)
    o2 = s["o"].view(T, Hq * d)
    do = api.gemm_bf16(dx2, w_o, b_mn=True, out_dtype=bf)
    dw_o = api.gemm_bf16(dx2, o2, a_mn=True, b_mn=True, out_dtype=f32)
    dq, dk, dv = api.grouped_attn_bwd(layout, s["q"].view(T, Hq, d), s["k"].view(T, Hkv, d),
                                      s["v"].view(T, Hkv, d), s["o"], s["lse"],
                                      do.view(T, Hq, d), rope_theta=rope_theta,
                                      flags=s["attn_flags"], workspace=s["attn_ws"])
    dq, dk, dv = dq.view(T, Hq * d), dk.view(T, Hkv * d), dv.view(T, Hkv * d)
    dh1 = api.gemm_bf16(dq, wq, b_mn=True, out_dtype=f32)
    api.gemm_bf16(dk, wk, b_mn=True, out=dh1, accumulate=True)
    api.gemm_bf16(dv, wv, b_mn=True, out=dh1, accumulate=True)
    dw_qkv = torch.empty(w_qkv.shape, dtype=f32, device=x.device)
    dwq, dwk, dwv = _views(dw_qkv, Hq, Hkv, d)
    api.gemm_bf16(dq, s["h1"], a_mn=True, b_mn=True, out=dwq)
    api.gemm_bf16(dk, s["h1"], a_mn=True, b_mn=True, out=dwk)
    api.gemm_bf16(dv, s["h1"], a_mn=True, b_mn=True, out=dwv)
    dx, dg1 = api.rmsnorm_bwd(x, g1, s["r1"], dh1, dres=dx2, dx_dtype=bf)
    return LayerGrads(dx, dw_qkv, dw_o, dw_gu, dw_d, dg1, dg2)
