"""CPU oracle for one Llama-style decoder layer over packed shared-prefix groups.
TEST INFRASTRUCTURE ONLY: used by the tests, never by the library or its binding.

The layer (RMSNorm, Q/K/V projections, RoPE, grouped attention, output projection, residual,
RMSNorm, SwiGLU MLP, residual) is computed the way the repeated-prefix baseline computes it: every
[P; Ri] of a group runs through the whole layer on its own (positions 0 .. Lp + ri - 1), with an
explicit backward.  The packed results follow the same mapping as the attention oracle: suffix rows
from their copy, prefix rows of y from copy 0, prefix rows of dx summed over the copies with the
upstream dy of prefix rows routed into copy 0, and every weight gradient summed over all copies'
tokens.  The abstract page of Prefix Grouper claims identical outputs and gradients for the packed
computation; the Pith review ("major comments", Appendix A.1 objection) asks exactly for the
parameter gradients to match, which the tests check through the second formulation here
(``layer_packed``: one pass over the packed sequence with the dense grouped mask).

Readings: RMSNorm without mean subtraction, eps inside the square root, gains multiplied after
normalisation; SwiGLU = silu(gate) * up with gate the first half of the gate/up projection; no
biases; softmax scale d^-1/2; RoPE, GQA head mapping and masks as in prefix_grouper_oracle.
Everything in float64 with plain PyTorch CPU ops.  Pinned by tests against torch autograd of
torch.nn.functional routines (G = 1), and by layer_packed == layer_repeated.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

from . import prefix_grouper_oracle as orc

F64 = torch.float64


@dataclasses.dataclass
class LayerResult:
    y: torch.Tensor
    dx: torch.Tensor
    w_qkv: torch.Tensor
    w_o: torch.Tensor
    w_gu: torch.Tensor
    w_d: torch.Tensor
    g1: torch.Tensor
    g2: torch.Tensor


def rmsnorm(x, g, eps):
    rstd = torch.rsqrt((x * x).mean(dim=-1) + eps)
    return x * rstd[:, None] * g[None, :], rstd


def rmsnorm_vjp(x, g, rstd, dout):
    yh = x * rstd[:, None]
    gd = g[None, :] * dout
    dx = rstd[:, None] * (gd - yh * (yh * gd).mean(dim=-1, keepdim=True))
    return dx, (dout * yh).sum(dim=0)


def _split_w(w_qkv, Hq, Hkv, d):
    nq, nk = Hq * d, Hkv * d
    return w_qkv[:nq], w_qkv[nq:nq + nk], w_qkv[nq + nk:]


class _Layer:
    """Forward/backward of the layer on one sequence whose attention is given by `attn`."""

    def __init__(self, W, Hq, Hkv, d, theta, eps):
        self.w_qkv, self.w_o, self.w_gu, self.w_d, self.g1, self.g2 = (t.to(F64) for t in W)
        self.Hq, self.Hkv, self.d, self.theta, self.eps = Hq, Hkv, d, theta, eps

    def run(self, x, dy, attn_fwd, attn_bwd):
        Hq, Hkv, d = self.Hq, self.Hkv, self.d
        n = x.shape[0]
        wq, wk, wv = _split_w(self.w_qkv, Hq, Hkv, d)
        h1, r1 = rmsnorm(x, self.g1, self.eps)
        q = (h1 @ wq.T).view(n, Hq, d)
        k = (h1 @ wk.T).view(n, Hkv, d)
        v = (h1 @ wv.T).view(n, Hkv, d)
        o, saved = attn_fwd(q, k, v)
        o2 = o.reshape(n, Hq * d)
        x2 = x + o2 @ self.w_o.T
        h2, r2 = rmsnorm(x2, self.g2, self.eps)
        gu = h2 @ self.w_gu.T
        I = gu.shape[1] // 2
        g, u = gu[:, :I], gu[:, I:]
        sg = torch.sigmoid(g)
        act = g * sg * u
        y = x2 + act @ self.w_d.T
        # backward
        d_act = dy @ self.w_d
        dw_d = dy.T @ act
        dg = d_act * u * sg * (1 + g * (1 - sg))
        du = d_act * g * sg
        dgu = torch.cat([dg, du], dim=1)
        dh2 = dgu @ self.w_gu
        dw_gu = dgu.T @ h2
        dx2, dg2 = rmsnorm_vjp(x2, self.g2, r2, dh2)
        dx2 = dx2 + dy
        do = (dx2 @ self.w_o).view(n, Hq, d)
        dw_o = dx2.T @ o2
        dq, dk, dv = attn_bwd(saved, do)
        dq, dk, dv = dq.reshape(n, -1), dk.reshape(n, -1), dv.reshape(n, -1)
        dh1 = dq @ wq + dk @ wk + dv @ wv
        dw_qkv = torch.cat([dq.T @ h1, dk.T @ h1, dv.T @ h1], dim=0)
        dx, dg1 = rmsnorm_vjp(x, self.g1, r1, dh1)
        dx = dx + dx2
        return y, LayerResult(y, dx, dw_qkv, dw_o, dw_gu, dw_d, dg1, dg2)


def _causal_attention(Hq, Hkv, d, theta, pos):
    scale = d ** -0.5
    n = pos.numel()
    mfn = orc.causal_mask_fn(n)

    def fwd(q, k, v):
        qr, kr = orc.rope_rotate(q, pos, theta), orc.rope_rotate(k, pos, theta)
        o = torch.empty_like(q)
        lses = []
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            o[:, h], lse = orc.masked_attention_fwd(qr[:, h], kr[:, kh], v[:, kh], mfn, scale)
            lses.append(lse)
        return o, (qr, kr, v, o, lses)

    def bwd(saved, do):
        qr, kr, v, o, lses = saved
        dqr = torch.empty_like(qr)
        dkr = torch.zeros_like(kr)
        dv = torch.zeros_like(v)
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            a, b, c = orc.masked_attention_bwd(qr[:, h], kr[:, kh], v[:, kh], o[:, h], lses[h],
                                               do[:, h], mfn, scale)
            dqr[:, h] = a
            dkr[:, kh] += b
            dv[:, kh] += c
        return orc.rope_rotate_vjp(dqr, pos, theta), orc.rope_rotate_vjp(dkr, pos, theta), dv

    return fwd, bwd


def layer_repeated(prefix_lens, group_sizes, suffix_lens, x, dy, W, *, heads_q, heads_kv,
                   head_dim, theta, eps) -> LayerResult:
    """The layer computed copy by copy (repeated-prefix baseline), mapped onto packed rows.
    W = (w_qkv, w_o, w_gu, w_d, g1, g2)."""
    lay = orc.pack_layout(prefix_lens, group_sizes, suffix_lens)
    x, dy = x.to(F64), dy.to(F64)
    layer = _Layer(W, heads_q, heads_kv, head_dim, theta, eps)
    T = lay.total_tokens
    Y = torch.full_like(x, float("nan"))
    DX = torch.zeros_like(x)
    acc = None
    for b in range(len(prefix_lens)):
        lp = prefix_lens[b]
        segs = orc.group_segments(lay, b)
        copies = segs if segs else [None]
        for ci, i in enumerate(copies):
            rows = orc.baseline_rows(lay, b, i)
            n = rows.numel()
            if n == 0:
                continue
            pos = torch.arange(n)
            dyc = dy[rows].clone()
            if ci > 0:
                dyc[:lp] = 0          # upstream gradient of prefix rows routed into copy 0
            fwd, bwd = _causal_attention(heads_q, heads_kv, head_dim, theta, pos)
            y, res = layer.run(x[rows], dyc, fwd, bwd)
            if ci == 0:
                Y[rows[:lp]] = y[:lp]
            Y[rows[lp:]] = y[lp:]
            DX[rows] += res.dx
            if acc is None:
                acc = [res.w_qkv, res.w_o, res.w_gu, res.w_d, res.g1, res.g2]
            else:
                for a, g in zip(acc, [res.w_qkv, res.w_o, res.w_gu, res.w_d, res.g1, res.g2]):
                    a += g
    return LayerResult(Y, DX, *acc)


def layer_packed(prefix_lens, group_sizes, suffix_lens, x, dy, W, *, heads_q, heads_kv,
                 head_dim, theta, eps) -> LayerResult:
    """Second formulation: one pass over the packed sequence, grouped attention by dense mask."""
    lay = orc.pack_layout(prefix_lens, group_sizes, suffix_lens)
    x, dy = x.to(F64), dy.to(F64)
    layer = _Layer(W, heads_q, heads_kv, head_dim, theta, eps)

    def fwd(q, k, v):
        res = orc.packed_dense(lay, q, k, v, theta=theta)
        return res.o, (q, k, v)

    def bwd(saved, do):
        q, k, v = saved
        res = orc.packed_dense(lay, q, k, v, do, theta=theta)
        return res.dq, res.dk, res.dv

    _, res = layer.run(x, dy, fwd, bwd)
    return res
