"""GPU test helpers: the oracle side of a comparison, and pool-tile decoding.

Placement of a workload in paged pools lives in the package
(disaggregated_kv_attention_gb300.paged); the oracle, in contrast, reads the
logical tensors directly, so a paging mistake shows up as a parity failure.
"""
from __future__ import annotations

import os
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from disaggregated_kv_attention_gb300 import workload as wl
from disaggregated_kv_attention_gb300.paged import Placed, params, place  # noqa: F401


def _np(t):
    return t.to(torch.float64).numpy()


def oracle(w: wl.Workload, agents: Sequence[int], q_heads: Optional[Sequence[int]] = None,
           q_rows: Optional[Sequence[int]] = None) -> Dict[int, np.ndarray]:
    """fp64 oracle outputs {agent: [q_len or len(q_rows), Hq, D]} (NaN outside q_heads)."""
    from oracle import residual_attention as ra
    res = {}
    for a in agents:
        kb, vb = w.agent_base(a)
        q = _np(w.q[a])
        pos = w.positions[a].numpy()
        if q_rows is not None:
            q, pos = q[list(q_rows)], pos[list(q_rows)]
        res[a] = ra.residual_attention(q, pos, _np(kb), _np(vb), _np(w.k_res[a]), _np(w.v_res[a]),
                                       _np(w.B_k[a]), _np(w.B_v[a]), w.cfg.rope_theta, q_heads=q_heads)
    return res


# (test id, max_abs, rel_l2) of every comparison made in this process; the session summary
# (tests/conftest.py) prints them so that a drift towards the tolerance shows in the log.
PARITY_LOG: List[tuple] = []


def record(m: dict) -> None:
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    PARITY_LOG.append((test, m["max_abs"], m["rel_l2"]))


def compare(out: torch.Tensor, ref: Dict[int, np.ndarray], q_rows: Optional[Sequence[int]] = None):
    from oracle import residual_attention as ra
    got, want = [], []
    for a, r in ref.items():
        o = out[a].to(torch.float64).cpu().numpy()
        if q_rows is not None:
            o = o[list(q_rows)]
        got.append(o)
        want.append(r)
    got, want = np.stack(got), np.stack(want)
    m = ra.metrics(got, want)
    record(m)
    return m, ra.within_tolerance(got, want)


# base tile / residual tile decoding, from the layout documented in include/forkkv.h
def base_tile_rows(tile: np.ndarray) -> np.ndarray:
    """[4096] uint8 -> [16, 128] uint16 (bf16 bit patterns), logical row order."""
    out = np.empty((16, 128), np.uint16)
    u16 = tile.view(np.uint16)
    for t in range(16):
        for d in range(128):
            off = (d // 64) * 2048 + t * 128 + ((((d % 64) // 8) ^ (t % 8)) * 16) + (d % 8) * 2
            out[t, d] = u16[off // 2]
    return out


def res_tile_rows(tile: np.ndarray) -> np.ndarray:
    out = np.empty((16, 16), np.uint16)
    u16 = tile.view(np.uint16)
    for t in range(16):
        for k in range(16):
            off = t * 32 + (((k // 8) ^ ((t // 4) % 2)) * 16) + (k % 8) * 2
            out[t, k] = u16[off // 2]
    return out
