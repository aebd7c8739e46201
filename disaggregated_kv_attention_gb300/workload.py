"""Seeded synthetic workloads shaped like multi-agent fork fan-outs.

This module only draws numbers: it holds none of the attention arithmetic, so
that the fp64 oracle and the CUDA path can both be fed from it without sharing
any computation.

Workload shapes follow the ForkKV L2 digest, section 2 (Q2: a shared base
cache of xW rows plus a per-agent rank-r residual xA_i) and section 3 (agents
forked from a shared prefix, each appending private tokens).  Distributions:
base rows, residual rows and q are N(0, 1); the adapter up-projections B_k and
B_v are N(0, 0.02); every draw is made in fp32 by a CPU ``torch.Generator`` and
rounded to bf16 (round to nearest even).

Draw order (fixed, so a seed defines the workload):
  1. lengths of every node with a drawn length, in node order;
  2. base rows (K then V) of every shared node, in node order;
  3. base rows (K then V) of every agent's private suffix, in agent order;
  4. residual rows (k_res then v_res) of every agent over its whole sequence;
  5. q;  6. B_k of every agent;  7. B_v of every agent.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence, Tuple

import torch

HEAD_DIM = 128
RANK = 16
PAGE_SIZE = 16


@dataclasses.dataclass(frozen=True)
class Node:
    """A node of the fork tree: a run of tokens appended after its parent's."""

    name: str
    parent: int                 # index of the parent node, -1 for the root
    tokens: Tuple[int, int]     # inclusive (lo, hi); lo == hi means fixed
    agent: bool                 # leaves are agents


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    index: int                  # seed = 1000 + index
    n_q_heads: int
    n_kv_heads: int
    rope_theta: float
    model_layers: int           # layer count of the model the shape is taken from
    q_len: int                  # 1 for decode, C for a prefill chunk
    nodes: Tuple[Node, ...]
    head_dim: int = HEAD_DIM
    rank: int = RANK
    page_size: int = PAGE_SIZE
    description: str = ""
    hidden: int = 4096          # model hidden size (inputs of the k/v projections; the residual fill's K)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def seed(self) -> int:
        return 1000 + self.index

    @property
    def agent_nodes(self) -> List[int]:
        return [i for i, n in enumerate(self.nodes) if n.agent]

    @property
    def n_agents(self) -> int:
        return len(self.agent_nodes)


def _fan(root_tokens: int, n_agents: int, suffix: Tuple[int, int]) -> Tuple[Node, ...]:
    nodes = [Node("root", -1, (root_tokens, root_tokens), False)]
    nodes += [Node(f"agent{i}", 0, suffix, True) for i in range(n_agents)]
    return tuple(nodes)


def _two_level(root_tokens, n_trunks, trunk_tokens, per_trunk, suffix) -> Tuple[Node, ...]:
    nodes = [Node("root", -1, (root_tokens, root_tokens), False)]
    trunks = []
    for t in range(n_trunks):
        trunks.append(len(nodes))
        nodes.append(Node(f"trunk{t}", 0, (trunk_tokens, trunk_tokens), False))
    for t in range(n_trunks):
        for i in range(per_trunk):
            nodes.append(Node(f"agent{t}_{i}", trunks[t], suffix, True))
    return tuple(nodes)


CONFIGS: Dict[str, WorkloadConfig] = {
    c.name: c
    for c in [
        WorkloadConfig(
            "tiny_decode", 0, 32, 8, 500000.0, 1, 1, _fan(512, 4, (64, 64)),
            description="32q/8kv, 4 agents on a 512-token prefix + 64 private tokens each, 1 query/agent"),
        WorkloadConfig(
            "llama3_8b_decode", 1, 32, 8, 500000.0, 32, 1, _fan(8192, 8, (256, 1024)),
            description="32q/8kv, 8 agents on an 8192-token prefix (refcount 8) + U[256,1024] private tokens, 1 query/agent",
            hidden=4096),
        WorkloadConfig(
            "qwen25_7b_mapreduce_decode", 2, 28, 4, 1000000.0, 28, 1, _fan(32768, 32, (64, 4096)),
            description="28q/4kv, 32 agents on a 32768-token prefix + U[64,4096] private tokens, 1 query/agent",
            hidden=3584),
        WorkloadConfig(
            "qwen25_14b_prefill", 3, 40, 8, 1000000.0, 48, 2048, _fan(16384, 8, (2048, 2048)),
            description="40q/8kv, 8 agents each prefilling a causal 2048-token chunk on a 16384-token prefix",
            hidden=5120),
        WorkloadConfig(
            "llama3_70b_stress_decode", 4, 64, 8, 500000.0, 80, 1,
            _two_level(131072, 4, 8192, 16, (1, 4096)),
            description="64q/8kv, 64 agents: 131072-token root -> 4 trunks of 8192 -> 16 agents each with U[1,4096] private tokens",
            hidden=8192),
    ]
}

CONFIG_ORDER = [
    "tiny_decode", "llama3_8b_decode", "qwen25_7b_mapreduce_decode",
    "qwen25_14b_prefill", "llama3_70b_stress_decode",
]


@dataclasses.dataclass
class Workload:
    """Logical (unpaged) tensors of one seeded workload, all bf16 on the CPU."""

    cfg: WorkloadConfig
    node_tokens: List[int]                 # drawn length of every node
    node_start: List[int]                  # first logical position of every node
    node_k: List[Optional[torch.Tensor]]   # [n_tokens, Hkv, D] base K rows (already rotated)
    node_v: List[Optional[torch.Tensor]]   # [n_tokens, Hkv, D] base V rows
    k_res: List[torch.Tensor]              # per agent [L_a, r]
    v_res: List[torch.Tensor]              # per agent [L_a, r]
    q: torch.Tensor                        # [A, q_len, Hq, D]
    B_k: torch.Tensor                      # [A, r, Hkv*D]
    B_v: torch.Tensor                      # [A, r, Hkv*D]
    seq_lens: torch.Tensor                 # [A] int32, includes the query tokens
    positions: torch.Tensor                # [A, q_len] int32 absolute query positions

    @property
    def n_agents(self) -> int:
        return self.cfg.n_agents

    def agent_path(self, a: int) -> List[int]:
        """Node indices from the root down to agent a's leaf."""
        node = self.cfg.agent_nodes[a]
        path = []
        while node >= 0:
            path.append(node)
            node = self.cfg.nodes[node].parent
        return path[::-1]

    def agent_base(self, a: int) -> Tuple[torch.Tensor, torch.Tensor]:
        """Agent a's base K and V rows over its whole sequence (concatenation)."""
        path = self.agent_path(a)
        k = torch.cat([self.node_k[i] for i in path], dim=0)
        v = torch.cat([self.node_v[i] for i in path], dim=0)
        return k, v


def _randn(g: torch.Generator, shape: Sequence[int], std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def generate(cfg: WorkloadConfig, seed: Optional[int] = None, b_std: float = 0.02) -> Workload:
    """Draw the logical tensors of ``cfg`` (see the module docstring for the order)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(cfg.seed if seed is None else seed)
    nodes = cfg.nodes
    Hkv, D, r = cfg.n_kv_heads, cfg.head_dim, cfg.rank

    # 1. lengths
    node_tokens = []
    for n in nodes:
        lo, hi = n.tokens
        if lo == hi:
            node_tokens.append(lo)
        else:
            node_tokens.append(int(torch.randint(lo, hi + 1, (1,), generator=g).item()))
    node_start = []
    for i, n in enumerate(nodes):
        node_start.append(0 if n.parent < 0 else node_start[n.parent] + node_tokens[n.parent])

    node_k: List[Optional[torch.Tensor]] = [None] * len(nodes)
    node_v: List[Optional[torch.Tensor]] = [None] * len(nodes)
    # 2. shared rows
    for i, n in enumerate(nodes):
        if not n.agent:
            node_k[i] = _randn(g, (node_tokens[i], Hkv, D))
            node_v[i] = _randn(g, (node_tokens[i], Hkv, D))
    # 3. private rows
    agents = cfg.agent_nodes
    for i in agents:
        node_k[i] = _randn(g, (node_tokens[i], Hkv, D))
        node_v[i] = _randn(g, (node_tokens[i], Hkv, D))
    seq_lens = [node_start[i] + node_tokens[i] for i in agents]
    # 4. residual rows
    k_res, v_res = [], []
    for L in seq_lens:
        k_res.append(_randn(g, (L, r)))
        v_res.append(_randn(g, (L, r)))
    # 5. q
    A = len(agents)
    q = _randn(g, (A, cfg.q_len, cfg.n_q_heads, D))
    # 6, 7. adapters
    B_k = _randn(g, (A, r, Hkv * D), b_std)
    B_v = _randn(g, (A, r, Hkv * D), b_std)

    lens = torch.tensor(seq_lens, dtype=torch.int32)
    pos = lens[:, None] - cfg.q_len + torch.arange(cfg.q_len, dtype=torch.int32)[None, :]
    return Workload(cfg, node_tokens, node_start, node_k, node_v, k_res, v_res, q, B_k, B_v,
                    lens, pos.to(torch.int32))


def custom_config(name: str, n_q_heads: int, n_kv_heads: int, nodes: Sequence[Node],
                  q_len: int = 1, rope_theta: float = 500000.0, index: int = 100) -> WorkloadConfig:
    """A small ad-hoc workload (tests: ragged tails, single keys, deep trees)."""
    return WorkloadConfig(name, index, n_q_heads, n_kv_heads, rope_theta, 1, q_len, tuple(nodes))
