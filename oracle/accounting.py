"""Closed-form memory and page-count formulas (test infrastructure only).

* ForkKV L2, section 4 (memory ratio): one shared base of s tokens x n
  dimensions plus N residuals of s x r, against N unified caches of s x n:
  M_R = (s n + N s r) / (N s n) = 1/N + r/n.
* ForkServe README, "Design vs APC" / "Methods": live KV of a fan-out with trunk
  L and residuals l_i is b(L + sum l_i) under copy-on-write and b(kL + sum l_i)
  when every child clones the trunk.
* ForkServe README, unaligned tail: with r = L mod P, the pack path costs
  k ceil((r + l)/P) child pages; the freeze path 1 + k ceil(l/P).
"""
from __future__ import annotations

from typing import Sequence


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def memory_ratio(n_agents: int, rank: int, width: int) -> float:
    """M_R = 1/N + r/n."""
    return 1.0 / n_agents + rank / width


def memory_ratio_from_sizes(tokens: int, width: int, n_agents: int, rank: int) -> float:
    """M_R from the sizes themselves: (s n + N s r) / (N s n)."""
    return (tokens * width + n_agents * tokens * rank) / (n_agents * tokens * width)


def m_cow(bytes_per_token: int, trunk: int, residuals: Sequence[int]) -> int:
    return bytes_per_token * (trunk + sum(residuals))


def m_clone(bytes_per_token: int, trunk: int, residuals: Sequence[int]) -> int:
    return bytes_per_token * (len(residuals) * trunk + sum(residuals))


def pages_clone(trunk: int, k: int, residual: int, page: int) -> int:
    """Every child holds its own copy of trunk + residual (content-addressed miss)."""
    return k * ceil_div(trunk + residual, page)


def pages_pack_children(trunk: int, k: int, residual: int, page: int) -> int:
    """Child pages on the pack path: the r = L mod P tail rows are cloned into each child."""
    return k * ceil_div(trunk % page + residual, page)


def pages_freeze_children(trunk: int, k: int, residual: int, page: int) -> int:
    """One read-only shared tail page plus every child's private residual pages."""
    return 1 + k * ceil_div(residual, page)


def pages_fork_pack(trunk: int, k: int, residual: int, page: int) -> int:
    """Live base pages of a fan-out on the pack path: the trunk once, plus child pages."""
    return ceil_div(trunk, page) + pages_pack_children(trunk, k, residual, page)


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int = 2) -> int:
    """K and V of every layer for one token (a unified, or a base, cache row)."""
    return layers * 2 * kv_heads * head_dim * elem_bytes


def residual_bytes_per_token(layers: int, rank: int, elem_bytes: int = 2) -> int:
    """xA_k and xA_v of every layer for one token (a residual cache row)."""
    return layers * 2 * rank * elem_bytes
