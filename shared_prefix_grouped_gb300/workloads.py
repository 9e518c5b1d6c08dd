"""Seeded synthetic workloads for grouped attention over packed [P; R1; ...; RG] sequences.

This module only draws numbers: suffix lengths and the Q/K/V/dO tensors, in the shapes and
distributions of the long-prefix GRPO workloads the Prefix Grouper pages describe (abstract page:
long shared prefixes; skill page "prefix-grouper-grpo", Practical Guidance: prefix much longer than
the responses, G typically 4-8).  It holds none of the method's arithmetic, so the CUDA path and the
CPU oracle can both take their inputs from here without sharing any computation.

Every draw uses a CPU ``torch.Generator`` seeded from the workload, in fp32, then a cast to the
workload's dtype (round-to-nearest-even for bf16).  Order of draws: suffix lengths, Q, K, V, dO.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One grouped-attention problem: B groups, each a shared prefix followed by G suffixes."""

    name: str
    dtype: str                       # "f32" or "bf16"
    num_groups: int                  # B
    group_size: int                  # G (suffixes per group)
    prefix_len: int                  # Lp (same for every group of a workload)
    heads_q: int                     # Hq
    heads_kv: int                    # Hkv (Hq % Hkv == 0; q-head h uses kv-head h // (Hq // Hkv))
    head_dim: int                    # d
    suffix_lens: Optional[tuple] = None   # fixed lengths (len B*G), or None to draw them
    suffix_range: Optional[tuple] = None  # (lo, hi) inclusive range for uniform draws
    rope_theta: float = 0.0          # 0 disables RoPE
    input_scale: float = 1.0         # Q, K, V are N(0,1) * input_scale; dO is N(0,1)
    seed: int = 1000
    responses_only: bool = False     # forward of the response rows only (scoring)


# Index 0 is the small fp32 case, 1..3 the bf16 fwd+bwd attention cases, 4 the forward-only
# scoring case: 16 candidate continuations of 1-4 tokens scored against one 32k-token context (the
# short-suffix shape in which grouped attention is bound by reading K/V, Pith review "Core claim").
# The decoder-layer workload is described by LayerWorkload below.
WORKLOADS: List[Workload] = [
    Workload("fp32_h2_d64_p256_g4", "f32", 1, 4, 256, 2, 2, 64,
             suffix_lens=(32, 48, 64, 16), rope_theta=0.0, seed=1000),
    Workload("bf16_mha_h32_d128_p4096_g8_r512", "bf16", 1, 8, 4096, 32, 32, 128,
             suffix_lens=(512,) * 8, rope_theta=1e4, input_scale=128 ** -0.5, seed=1001),
    Workload("bf16_gqa32x8_d128_b8_p2048_g16_r64-512", "bf16", 8, 16, 2048, 32, 8, 128,
             suffix_range=(64, 512), rope_theta=1e4, seed=1002),
    Workload("bf16_gqa32x8_d128_p16384_g16_r256-1024", "bf16", 1, 16, 16384, 32, 8, 128,
             suffix_range=(256, 1024), rope_theta=5e5, seed=1003),
    Workload("bf16_gqa32x8_d128_p32768_g16_r1-4_score", "bf16", 1, 16, 32768, 32, 8, 128,
             suffix_range=(1, 4), rope_theta=5e5, seed=1005, responses_only=True),
]


@dataclasses.dataclass(frozen=True)
class LayerWorkload:
    """One Llama-style decoder layer over packed groups (random-init weights N(0, 0.02))."""

    name: str = "llama_layer_h4096_gqa32x8_mlp14336_b2_p8192_g8_r1024"
    hidden: int = 4096
    heads_q: int = 32
    heads_kv: int = 8
    head_dim: int = 128
    mlp: int = 14336
    num_groups: int = 2
    group_size: int = 8
    prefix_len: int = 8192
    suffix_len: int = 1024
    rope_theta: float = 5e5
    rms_eps: float = 1e-5
    weight_std: float = 0.02
    seed: int = 1004


def by_name(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def torch_dtype(dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def draw_suffix_lens(w: Workload, gen: torch.Generator) -> List[int]:
    """Suffix lengths for all B*G responses, group-major."""
    n = w.num_groups * w.group_size
    if w.suffix_lens is not None:
        assert len(w.suffix_lens) == n
        return [int(x) for x in w.suffix_lens]
    lo, hi = w.suffix_range
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


@dataclasses.dataclass
class Problem:
    """Host tensors of one drawn workload, in the packed token order."""

    workload: Workload
    prefix_lens: List[int]           # per group
    group_sizes: List[int]           # per group
    suffix_lens: List[int]           # per response, group-major
    q: torch.Tensor                  # [T, Hq, d]
    k: torch.Tensor                  # [T, Hkv, d]
    v: torch.Tensor                  # [T, Hkv, d]
    do: torch.Tensor                 # [T, Hq, d]

    @property
    def total_tokens(self) -> int:
        return sum(self.prefix_lens) + sum(self.suffix_lens)


def make_problem(w: Workload, *, suffix_lens: Optional[List[int]] = None,
                 prefix_lens: Optional[List[int]] = None,
                 group_sizes: Optional[List[int]] = None,
                 seed: Optional[int] = None) -> Problem:
    """Draw a problem.  Lengths may be overridden (edge cases); values are always drawn."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    drawn = draw_suffix_lens(w, gen)
    if suffix_lens is None:
        suffix_lens = drawn
    if group_sizes is None:
        group_sizes = [w.group_size] * w.num_groups
    if prefix_lens is None:
        prefix_lens = [w.prefix_len] * len(group_sizes)
    assert len(suffix_lens) == sum(group_sizes) and len(prefix_lens) == len(group_sizes)
    T = sum(prefix_lens) + sum(suffix_lens)
    dt = torch_dtype(w.dtype)

    def draw(heads, scale):
        x = torch.randn((T, heads, w.head_dim), generator=gen, dtype=torch.float32)
        if scale != 1.0:
            x = x * scale
        return x.to(dt)

    q = draw(w.heads_q, w.input_scale)
    k = draw(w.heads_kv, w.input_scale)
    v = draw(w.heads_kv, w.input_scale)
    do = draw(w.heads_q, 1.0)
    return Problem(w, list(prefix_lens), list(group_sizes), list(suffix_lens), q, k, v, do)


def small_variant(w: Workload, *, prefix_len: int, suffix_lens: List[int], num_groups: int = 1,
                  heads_q: Optional[int] = None, heads_kv: Optional[int] = None,
                  seed: Optional[int] = None) -> Workload:
    """The same dtype/head_dim/RoPE recipe at a size the oracle finishes in seconds."""
    g = len(suffix_lens) // num_groups
    return dataclasses.replace(
        w, name=w.name + "_small", num_groups=num_groups, group_size=g, prefix_len=prefix_len,
        suffix_lens=tuple(suffix_lens), suffix_range=None,
        heads_q=heads_q or w.heads_q, heads_kv=heads_kv or w.heads_kv,
        seed=w.seed if seed is None else seed)


@dataclasses.dataclass
class LayerProblem:
    """Host tensors of one decoder-layer problem (packed token order)."""

    workload: LayerWorkload
    prefix_lens: List[int]
    group_sizes: List[int]
    suffix_lens: List[int]
    x: torch.Tensor        # [T, hidden] bf16
    dy: torch.Tensor       # [T, hidden] bf16
    w_qkv: torch.Tensor    # [(Hq + 2 Hkv) d, hidden] bf16 (q rows, then k rows, then v rows)
    w_o: torch.Tensor      # [hidden, Hq d]
    w_gu: torch.Tensor     # [2 mlp, hidden] (gate rows, then up rows)
    w_d: torch.Tensor      # [hidden, mlp]
    g1: torch.Tensor       # [hidden] RMSNorm gains (ones)
    g2: torch.Tensor

    @property
    def total_tokens(self) -> int:
        return sum(self.prefix_lens) + sum(self.suffix_lens)


def make_layer_problem(w: LayerWorkload, *, prefix_lens=None, group_sizes=None, suffix_lens=None,
                       seed: Optional[int] = None) -> LayerProblem:
    """Weights N(0, weight_std) in bf16, RMSNorm gains one, inputs x and upstream dy N(0, 1)."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    if group_sizes is None:
        group_sizes = [w.group_size] * w.num_groups
    if prefix_lens is None:
        prefix_lens = [w.prefix_len] * len(group_sizes)
    if suffix_lens is None:
        suffix_lens = [w.suffix_len] * sum(group_sizes)
    T = sum(prefix_lens) + sum(suffix_lens)
    bf = torch.bfloat16

    def rnd(shape, std=1.0):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        return (x * std if std != 1.0 else x).to(bf)

    qkv = (w.heads_q + 2 * w.heads_kv) * w.head_dim
    w_qkv = rnd((qkv, w.hidden), w.weight_std)
    w_o = rnd((w.hidden, w.heads_q * w.head_dim), w.weight_std)
    w_gu = rnd((2 * w.mlp, w.hidden), w.weight_std)
    w_d = rnd((w.hidden, w.mlp), w.weight_std)
    x = rnd((T, w.hidden))
    dy = rnd((T, w.hidden))
    ones = torch.ones(w.hidden, dtype=bf)
    return LayerProblem(w, list(prefix_lens), list(group_sizes), list(suffix_lens), x, dy, w_qkv,
                        w_o, w_gu, w_d, ones, ones.clone())


def small_layer(**kw) -> LayerWorkload:
    """A decoder layer small enough for the CPU oracle (head_dim stays 128)."""
    base = dict(hidden=256, heads_q=2, heads_kv=1, head_dim=128, mlp=384, num_groups=2,
                group_size=3, prefix_len=150, suffix_len=70, rope_theta=5e5, seed=1104)
    base.update(kw)
    return LayerWorkload(name="llama_layer_small", **base)


@dataclasses.dataclass(frozen=True)
class TreeWorkload:
    """Nested prefixes: segments in depth-first preorder (parent -1 for a root), e.g. a shared
    context, several user turns below it and several sampled responses below each turn."""

    name: str
    dtype: str
    parent: tuple
    lens: tuple
    heads_q: int
    heads_kv: int
    head_dim: int
    rope_theta: float = 0.0
    seed: int = 1006


def multi_turn(context: int, turns: int, turn_len: int, responses: int, response_len: int):
    """(parent, lens) of one context, `turns` user turns below it, `responses` answers per turn."""
    parent, lens = [-1], [context]
    for _ in range(turns):
        t = len(parent)
        parent.append(0)
        lens.append(turn_len)
        for _ in range(responses):
            parent.append(t)
            lens.append(response_len)
    return tuple(parent), tuple(lens)


TREE_WORKLOADS: List[TreeWorkload] = [
    TreeWorkload("bf16_gqa32x8_d128_tree_p4096_t4x512_r4x256", "bf16",
                 *multi_turn(4096, 4, 512, 4, 256), 32, 8, 128, rope_theta=5e5, seed=1006),
]


def tree_by_name(name: str) -> TreeWorkload:
    for w in TREE_WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


@dataclasses.dataclass
class TreeProblem:
    workload: TreeWorkload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor

    @property
    def total_tokens(self) -> int:
        return sum(self.workload.lens)


def make_tree_problem(w: TreeWorkload, seed: Optional[int] = None) -> TreeProblem:
    """Q, K, V, dO ~ N(0, 1) in fp32, cast to the workload dtype; draw order Q, K, V, dO."""
    gen = torch.Generator().manual_seed(w.seed if seed is None else seed)
    T = sum(w.lens)
    dt = torch_dtype(w.dtype)

    def draw(heads):
        return torch.randn((T, heads, w.head_dim), generator=gen, dtype=torch.float32).to(dt)

    q, k, v, do = draw(w.heads_q), draw(w.heads_kv), draw(w.heads_kv), draw(w.heads_q)
    return TreeProblem(w, q, k, v, do)
