"""Closed-form work counts for grouped attention (used by the benchmark to turn time into rates).

Visible (query, key) pairs of one head of one group with prefix Lp and responses r_1..r_G:
  grouped:  Lp(Lp+1)/2 + sum_i [ r_i * Lp + r_i(r_i+1)/2 ]
  repeated: sum_i (Lp + r_i)(Lp + r_i + 1)/2
The prefix rows are causal once; every response row sees the whole prefix and its own causal past.
The ratio grouped/repeated tends to 1/G as Lp/r grows (Lemma 2.2 of the paper, as summarised by the
Pith review of Prefix Grouper, "Core claim").

FLOPs follow the usual attention convention: 4 * d * pairs per head forward (QK^T and PV, two flops
per multiply-add), and the backward counted as 2.5x the forward, so forward+backward is
14 * d * pairs per head.
"""
from __future__ import annotations

from typing import Sequence


def group_pairs(prefix_len: int, suffix_lens: Sequence[int]) -> int:
    lp = prefix_len
    return lp * (lp + 1) // 2 + sum(r * lp + r * (r + 1) // 2 for r in suffix_lens)


def group_repeated_pairs(prefix_len: int, suffix_lens: Sequence[int]) -> int:
    if len(suffix_lens) == 0:
        return prefix_len * (prefix_len + 1) // 2
    return sum((prefix_len + r) * (prefix_len + r + 1) // 2 for r in suffix_lens)


def split_groups(group_sizes: Sequence[int], suffix_lens: Sequence[int]):
    out, k = [], 0
    for g in group_sizes:
        out.append(list(suffix_lens[k:k + g]))
        k += g
    return out


def total_pairs(prefix_lens, group_sizes, suffix_lens) -> int:
    return sum(group_pairs(lp, rs) for lp, rs in zip(prefix_lens, split_groups(group_sizes, suffix_lens)))


def total_repeated_pairs(prefix_lens, group_sizes, suffix_lens) -> int:
    return sum(group_repeated_pairs(lp, rs)
               for lp, rs in zip(prefix_lens, split_groups(group_sizes, suffix_lens)))


def attn_flops(pairs: int, heads_q: int, head_dim: int, phase: str = "fwdbwd") -> float:
    per = 4.0 * head_dim * pairs * heads_q
    return {"fwd": per, "bwd": 2.5 * per, "fwdbwd": 3.5 * per}[phase]


def repeated_tokens(prefix_lens, group_sizes, suffix_lens) -> int:
    total = 0
    for lp, rs in zip(prefix_lens, split_groups(group_sizes, suffix_lens)):
        total += lp + sum(rs) + lp * (max(len(rs), 1) - 1)
    return total
