"""The stated tolerance detects every plausible kernel mistake.

A mistake is planted on the CPU, by recomposing the oracle's own steps with one
step changed; each such output must FAIL the tolerance (max abs <= 2e-2 and
relative L2 <= 5e-3) against the true oracle, on the tiny workload and on a
long one.  If a mutation passed, a GPU kernel carrying that bug could pass the
parity tests.
"""
import math

import numpy as np
import pytest
import torch

from oracle import residual_attention as ra
from disaggregated_kv_attention_gb300 import workload as wl

D = 128


def _np(t):
    return t.to(torch.float64).numpy()


def _rope_interleaved(x, pos, theta):
    f = theta ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    ang = np.asarray(pos, float)[:, None] * f[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[:, 0::2], x[:, 1::2]
    out = np.empty_like(x)
    out[:, 0::2] = a * c - b * s
    out[:, 1::2] = b * c + a * s
    return out


def _compose(w, a, heads, mutation=None):
    """Oracle steps recomposed for agent a, with at most one step changed."""
    cfg = w.cfg
    theta, G = cfg.rope_theta, cfg.group
    kb, vb = w.agent_base(a)
    kb, vb = _np(kb), _np(vb)
    L = kb.shape[0]
    kr, vr = _np(w.k_res[a]), _np(w.v_res[a])
    Bk, Bv = _np(w.B_k[a]), _np(w.B_v[a])
    q = _np(w.q[a])
    qpos = w.positions[a].numpy()
    kpos = np.arange(L)
    vis = kpos[None, :] <= qpos[:, None]
    if mutation == "mask_drops_current_key":
        vis = kpos[None, :] < qpos[:, None]
    scale = 1 / math.sqrt(D)
    if mutation == "softmax_scale_1_over_D":
        scale = 1 / D
    out = np.full(q.shape, np.nan)
    for h in sorted({hq // G for hq in heads}):
        hb = (h + 1) % cfg.n_kv_heads if mutation == "B_slice_of_wrong_head" else h
        U = kr @ ra.head_slice(Bk, hb, D)
        if mutation == "no_rope_on_k_lora":
            K_lora = U
        elif mutation == "rope_at_page_offset":
            K_lora = ra.rope_rotate_half(U, kpos % 16, theta)
        elif mutation == "rope_positions_restart_at_suffix":
            start = w.node_start[w.cfg.agent_nodes[a]]
            K_lora = ra.rope_rotate_half(U, np.where(kpos >= start, kpos - start, kpos), theta)
        elif mutation == "interleaved_rope_pairs":
            K_lora = _rope_interleaved(U, kpos, theta)
        else:
            K_lora = ra.rope_rotate_half(U, kpos, theta)
        if mutation == "drop_k_lora":
            K_lora = 0 * K_lora
        K = kb[:, h] + K_lora
        V_lora = vr @ ra.head_slice(Bv, hb, D)
        if mutation == "drop_v_lora":
            V_lora = 0 * V_lora
        V = vb[:, h] + V_lora
        for hq in heads:
            if hq // G == h:
                out[:, hq] = ra.softmax_attention(q[:, hq], K, V, vis, scale)
    return out


def _online_without_residual_rescale(q_vec, pos, kb, vb, kr, vr, Bk, Bv, theta, scale, block=16):
    # the kernel's loop with acc_r NOT rescaled when the running max grows
    m, l = -np.inf, 0.0
    acc, acc_r = np.zeros(D), np.zeros(kr.shape[1])
    for j0 in range(0, kb.shape[0], block):
        j1 = min(kb.shape[0], j0 + block)
        p_idx = np.arange(j0, j1)
        vis = p_idx <= pos
        K = ra.residual_keys(kb[j0:j1], kr[j0:j1], Bk, p_idx, theta)
        s = np.where(vis, (K @ q_vec) * scale, -np.inf)
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m > -np.inf else 0.0
        p = np.where(vis, np.exp(s - m_new), 0.0)
        l = alpha * l + p.sum()
        acc = alpha * acc + p @ vb[j0:j1]
        acc_r = acc_r + p @ vr[j0:j1]
        m = m_new
    return (acc + acc_r @ Bv) / l


MUTATIONS = [
    "drop_k_lora", "drop_v_lora", "no_rope_on_k_lora", "rope_at_page_offset",
    "rope_positions_restart_at_suffix", "interleaved_rope_pairs", "B_slice_of_wrong_head",
    "mask_drops_current_key", "softmax_scale_1_over_D",
]

CASES = [("tiny_decode", None, None), ("llama3_8b_decode", [0, 3, 6], None)]


@pytest.fixture(scope="module")
def workloads():
    return {name: wl.generate(wl.CONFIGS[name]) for name, _, _ in CASES}


def _all(w, agents, fn):
    outs, refs = [], []
    for a in agents:
        ref = _compose(w, a, range(w.cfg.n_q_heads))
        outs.append(fn(a))
        refs.append(ref)
    return np.stack(outs), np.stack(refs)


@pytest.mark.parametrize("cfg_name,agents,_", CASES)
def test_recomposition_is_the_oracle(workloads, cfg_name, agents, _):
    w = workloads[cfg_name]
    for a in (agents or range(w.n_agents))[:2]:
        kb, vb = w.agent_base(a)
        ref = ra.residual_attention(_np(w.q[a]), w.positions[a].numpy(), _np(kb), _np(vb), _np(w.k_res[a]),
                                    _np(w.v_res[a]), _np(w.B_k[a]), _np(w.B_v[a]), w.cfg.rope_theta)
        assert np.allclose(_compose(w, a, range(w.cfg.n_q_heads)), ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("mutation", MUTATIONS)
@pytest.mark.parametrize("cfg_name,agents,_", CASES)
def test_mutation_fails_tolerance(workloads, cfg_name, agents, _, mutation):
    w = workloads[cfg_name]
    agents = agents or range(w.n_agents)
    out, ref = _all(w, agents, lambda a: _compose(w, a, range(w.cfg.n_q_heads), mutation))
    assert not ra.within_tolerance(out, ref), (mutation, ra.metrics(out, ref))


@pytest.mark.parametrize("cfg_name,agents,heads", [("tiny_decode", None, range(32)),
                                                   ("llama3_8b_decode", [0, 5], [0, 9, 18, 27])])
def test_missing_residual_rescale_fails_tolerance(workloads, cfg_name, agents, heads):
    w = workloads[cfg_name]
    theta, G = w.cfg.rope_theta, w.cfg.group
    outs, refs = [], []
    for a in agents or range(w.n_agents):
        kb, vb = w.agent_base(a)
        kb, vb = _np(kb), _np(vb)
        ref = _compose(w, a, heads)
        for hq in heads:
            h = hq // G
            outs.append(_online_without_residual_rescale(
                _np(w.q[a, 0, hq]), int(w.positions[a, 0]), kb[:, h], vb[:, h], _np(w.k_res[a]),
                _np(w.v_res[a]), ra.head_slice(_np(w.B_k[a]), h, D), ra.head_slice(_np(w.B_v[a]), h, D),
                theta, 1 / math.sqrt(D)))
            refs.append(ref[0, hq])
    out, ref = np.stack(outs), np.stack(refs)
    assert not ra.within_tolerance(out, ref), ra.metrics(out, ref)
