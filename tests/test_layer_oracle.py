"""Pins for the decoder-layer oracle: a single response (G = 1) against torch autograd of
torch.nn.functional routines; the copy-by-copy (repeated-prefix) layer against the packed
dense-mask layer, outputs and every parameter gradient (Pith review, Appendix A.1 objection: the
parameter gradients of the two computations must match)."""
import pytest
import torch
import torch.nn.functional as F

from oracle import layer_oracle as lo

F64 = torch.float64


def weights(H, Hq, Hkv, d, I, seed):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(s, generator=g, dtype=F64) * 0.3
    return (r((Hq + 2 * Hkv) * d, H), r(H, Hq * d), r(2 * I, H), r(H, I),
            1 + 0.1 * r(H), 1 + 0.1 * r(H))


def rope_complex(x, pos, theta):
    d = x.shape[-1]
    freq = theta ** (-(torch.arange(0, d, 2, dtype=F64)) / d)
    a = pos[:, None].to(F64) * freq[None, :]
    c, s = torch.cos(a)[:, None], torch.sin(a)[:, None]
    re, im = x[..., : d // 2], x[..., d // 2:]
    return torch.cat([re * c - im * s, re * s + im * c], dim=-1)


def torch_layer(x, W, Hq, Hkv, d, theta, eps):
    w_qkv, w_o, w_gu, w_d, g1, g2 = W
    n, H = x.shape
    nq, nk = Hq * d, Hkv * d
    h1 = F.rms_norm(x, (H,), weight=g1, eps=eps)
    q = F.linear(h1, w_qkv[:nq]).view(n, Hq, d)
    k = F.linear(h1, w_qkv[nq:nq + nk]).view(n, Hkv, d)
    v = F.linear(h1, w_qkv[nq + nk:]).view(n, Hkv, d)
    pos = torch.arange(n)
    q, k = rope_complex(q, pos, theta), rope_complex(k, pos, theta)
    rep = Hq // Hkv
    o = F.scaled_dot_product_attention(q.transpose(0, 1)[None],
                                       k.repeat_interleave(rep, 1).transpose(0, 1)[None],
                                       v.repeat_interleave(rep, 1).transpose(0, 1)[None],
                                       is_causal=True)[0].transpose(0, 1).reshape(n, nq)
    x2 = x + F.linear(o, w_o)
    h2 = F.rms_norm(x2, (H,), weight=g2, eps=eps)
    gu = F.linear(h2, w_gu)
    I = gu.shape[1] // 2
    return x2 + F.linear(F.silu(gu[:, :I]) * gu[:, I:], w_d)


def test_single_response_matches_torch_autograd():
    H, Hq, Hkv, d, I, theta, eps = 16, 2, 1, 8, 24, 50.0, 1e-5
    W = weights(H, Hq, Hkv, d, I, 1)
    g = torch.Generator().manual_seed(2)
    x = torch.randn((11, H), generator=g, dtype=F64)
    dy = torch.randn((11, H), generator=g, dtype=F64)
    res = lo.layer_repeated([7], [1], [4], x, dy, W, heads_q=Hq, heads_kv=Hkv, head_dim=d,
                            theta=theta, eps=eps)
    xx = x.clone().requires_grad_(True)
    WW = [w.clone().requires_grad_(True) for w in W]
    y = torch_layer(xx, WW, Hq, Hkv, d, theta, eps)
    (y * dy).sum().backward()
    assert torch.allclose(res.y, y.detach(), atol=1e-11)
    assert torch.allclose(res.dx, xx.grad, atol=1e-11)
    for got, w in zip([res.w_qkv, res.w_o, res.w_gu, res.w_d, res.g1, res.g2], WW):
        assert torch.allclose(got, w.grad, atol=1e-10)


@pytest.mark.parametrize("case", [
    ([6, 4], [2, 3], [3, 1, 2, 0, 5]),
    ([0, 5], [2, 1], [4, 2, 3]),
])
def test_repeated_layer_equals_packed_layer(case):
    plens, gsz, rs = case
    H, Hq, Hkv, d, I, theta, eps = 16, 4, 2, 4, 20, 30.0, 1e-5
    W = weights(H, Hq, Hkv, d, I, 3)
    T = sum(plens) + sum(rs)
    g = torch.Generator().manual_seed(4)
    x = torch.randn((T, H), generator=g, dtype=F64)
    dy = torch.randn((T, H), generator=g, dtype=F64)
    a = lo.layer_repeated(plens, gsz, rs, x, dy, W, heads_q=Hq, heads_kv=Hkv, head_dim=d,
                          theta=theta, eps=eps)
    b = lo.layer_packed(plens, gsz, rs, x, dy, W, heads_q=Hq, heads_kv=Hkv, head_dim=d,
                        theta=theta, eps=eps)
    for n in ["y", "dx", "w_qkv", "w_o", "w_gu", "w_d", "g1", "g2"]:
        assert torch.allclose(getattr(a, n), getattr(b, n), atol=1e-11, rtol=0), n
