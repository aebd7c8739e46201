"""Place a seeded fork-tree workload into paged device pools through the C ABI.

The fork tree is replayed with the library's allocator (root created, children
forked at their parent's full length, private tokens appended); copy-on-write
jobs run through forkkv_cow_copy_rows and every node's rows are scattered with
forkkv_write_rows.  Only slot indices (page * 16 + row) are computed here.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import forkkv as fk
from . import workload as wl


def token_slots(hole, start: int, n: int) -> np.ndarray:
    """Slots of tokens [start, start + n) of a sequence whose slot map is `hole` = (first hole slot,
    hole length), as include/forkkv.h defines them: token p sits in slot p, or p + hole length when the
    sequence has a hole and p is at or past its first slot."""
    p = np.arange(start, start + n, dtype=np.int64)
    hs, hn = int(hole[0]), int(hole[1])
    return np.where((hn > 0) & (p >= hs), p + hn, p)


def _slots(bpt_row: np.ndarray, start: int, n: int) -> np.ndarray:
    j = np.arange(start, start + n)
    return (bpt_row[j // 16].astype(np.int64) * 16 + (j % 16)).astype(np.int32)


class Placed:
    """Allocator handle, pools and device tensors of a placed workload."""


def place(w: wl.Workload, device="cuda", n_layers: int = 1, free_trunks: bool = True,
          slack_pages: int = 64) -> Placed:
    """Allocate, fill and describe the paged cache of workload ``w`` (layer 0 holds the data;
    further layers are byte copies of layer 0 at other addresses)."""
    cfg = w.cfg
    nodes = cfg.nodes
    Hkv = cfg.n_kv_heads
    n_base = sum(math.ceil(t / 16) + 2 for t in w.node_tokens) + slack_pages
    seq_len_node = [w.node_start[i] + w.node_tokens[i] for i in range(len(nodes))]
    n_res = sum(math.ceil(L / 16) + 1 for L in seq_len_node) + slack_pages
    alloc = fk.forkkv_alloc_create(n_base, n_res)
    pools = fk.Pools(n_base, n_res, Hkv, n_layers, device=device, fill=0)
    seq = [None] * len(nodes)
    jobs_all = []
    for i, n in enumerate(nodes):
        if n.parent < 0:
            seq[i] = fk.forkkv_seq_create(alloc, w.node_tokens[i])
        else:
            plen = seq_len_node[n.parent]
            seq[i], jobs = fk.forkkv_fork(alloc, seq[n.parent], plen)
            if jobs:
                fk.forkkv_cow_copy_rows(pools, jobs)  # parent's rows are already in place
                jobs_all += jobs
            jobs = fk.forkkv_append(alloc, seq[i], w.node_tokens[i])
            assert not jobs
        # this node's own base rows
        b, r, _ = fk.forkkv_page_tables(alloc, [seq[i]], math.ceil(seq_len_node[i] / 16))
        sl = torch.from_numpy(_slots(b[0], w.node_start[i], w.node_tokens[i])).to(device)
        kb = w.node_k[i].to(device).contiguous()
        vb = w.node_v[i].to(device).contiguous()
        fk.forkkv_write_rows(pools, 0, sl, None, kb, vb, None, None)
    agent_seqs = [seq[i] for i in cfg.agent_nodes]
    lens = [seq_len_node[i] for i in cfg.agent_nodes]
    stride = math.ceil(max(lens) / 16)
    bpt, rpt, lens_np = fk.forkkv_page_tables(alloc, agent_seqs, stride)
    assert list(lens_np) == lens == w.seq_lens.tolist()
    # every agent's residual rows over its whole sequence (private pages)
    for a in range(len(agent_seqs)):
        sl = torch.from_numpy(_slots(rpt[a], 0, lens[a])).to(device)
        fk.forkkv_write_rows(pools, 0, None, sl, None, None, w.k_res[a].to(device).contiguous(),
                             w.v_res[a].to(device).contiguous())
    if free_trunks:  # the agents' references must keep the shared pages alive
        for i, n in enumerate(nodes):
            if not n.agent:
                fk.forkkv_free(alloc, seq[i])
    for layer in range(1, n_layers):
        for t in (pools.k_base, pools.v_base, pools.k_res, pools.v_res):
            t[layer].copy_(t[0])
    P = Placed()
    P.alloc, P.pools, P.w = alloc, pools, w
    P.bpt_np, P.rpt_np = bpt, rpt
    P.bpt = torch.from_numpy(bpt).to(device)
    P.rpt = torch.from_numpy(rpt).to(device)
    P.seq_lens = w.seq_lens.to(device)
    P.positions = w.positions.to(device).contiguous()
    P.max_seq_len = int(max(lens))
    P.q = w.q.to(device).contiguous()
    P.B_k = w.B_k.to(device).contiguous()
    P.B_v = w.B_v.to(device).contiguous()
    P.jobs = jobs_all
    P.device = device
    return P


def params(P: Placed, out: torch.Tensor, layer: int = 0, use_plan: bool = True, rope: Optional[torch.Tensor] = None,
           target_ctas: int = 0, prefill: Optional[bool] = None):
    """forkkv_attn_params (+ the tensors it points to, kept alive in the returned dict)."""
    if prefill is None:
        prefill = P.w.cfg.q_len > 1
    keep = {}
    plan_t, info = None, None
    if use_plan and not prefill:
        plan, info = fk.forkkv_plan_build(P.bpt_np, P.w.seq_lens.numpy(), P.w.cfg.n_kv_heads, target_ctas)
        plan_t = torch.from_numpy(plan).to(P.device)
        keep["plan"] = plan_t
    p = fk.attn_params(P.pools, layer, P.q, out, P.bpt, P.rpt, P.seq_lens, P.positions, P.max_seq_len, P.B_k,
                       P.B_v, rope=rope, rope_theta=P.w.cfg.rope_theta, plan=plan_t, plan_info=info)
    keep["ws"] = fk.workspace_for(p, prefill=prefill, device=P.device)
    keep["info"] = info
    return p, keep
