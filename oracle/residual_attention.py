"""fp64 oracle for ResidualAttention (test infrastructure only).

What the method computes, restated from "ForkKV: Scaling Multi-LoRA Agent
Serving via Copy-on-Write Disaggregated KV Cache — L2":

* section 2 (Q2) and section 4 (reconstruction): a LoRA projection is
  xW + xA_i B_i, so the cache keeps the base part xW (shared, "bCache") apart
  from the rank-r residual xA_i (per agent, "rCache");
* section 3 (Figure 8) and section 7 (deferred RoPE): RoPE is already applied to
  the base keys, while the residual keys are stored unrotated; the rotation is
  applied after the up-projection K_res B_k, at each key's own position;
* section 4 (attention fusion) and section 7 (associativity): the value path
  is sum_j p_j V_base,j + (sum_j p_j V_res,j) B_v.

Because the method reaches the unified-cache attention exactly (up to rounding),
the oracle is that definition written out: it materialises

    K_j = Kb_j + RoPE_{p_j}(Kr_j B_k[:, hD:(h+1)D])
    V_j = Vb_j + Vr_j B_v[:, hD:(h+1)D]

per KV head h and runs textbook softmax attention over the keys a query may
see (key j visible iff p_j <= the query's position).

Readings where the pages are silent (each listed with its reason in the design
notes):
* RoPE is the rotate-half form: pairs (i, i + D/2) rotated by p * theta^(-2i/D),
  with no frequency scaling.
* Key positions are the keys' logical indices in the agent's sequence.
* q arrives already rotated; the softmax scale is 1/sqrt(D).
* One residual vector of rank r per token serves every KV head; the adapter
  B has r rows and Hkv*D columns and head h uses columns [hD, (h+1)D).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """Per-pair angular frequencies theta^(-2i/D), i < D/2 (rotate-half RoPE)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_rotate_half(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate rows of ``x`` [..., L, D] by their positions [L] (fp64).

    Pair (i, i + D/2) of a row at position p is turned by the angle p*f_i:
    (a, b) -> (a cos - b sin, b cos + a sin).
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    h = D // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(D, theta)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def residual_keys(k_base_h: np.ndarray, k_res: np.ndarray, B_k_h: np.ndarray,
                  key_positions: np.ndarray, theta: float) -> np.ndarray:
    """Unified keys of one KV head: K = Kb + RoPE(Kr @ B_k_h) (deferred RoPE)."""
    lora = np.asarray(k_res, np.float64) @ np.asarray(B_k_h, np.float64)
    return np.asarray(k_base_h, np.float64) + rope_rotate_half(lora, key_positions, theta)


def residual_values(v_base_h: np.ndarray, v_res: np.ndarray, B_v_h: np.ndarray) -> np.ndarray:
    """Unified values of one KV head: V = Vb + Vr @ B_v_h."""
    return np.asarray(v_base_h, np.float64) + np.asarray(v_res, np.float64) @ np.asarray(B_v_h, np.float64)


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, visible: np.ndarray,
                      sm_scale: float) -> np.ndarray:
    """Textbook attention: softmax(q K^T * scale) over the visible keys, times V.

    q [Nq, D], K [L, D], V [L, Dv], visible [Nq, L] (bool).  Every query must
    see at least one key.
    """
    if not np.all(visible.any(axis=1)):
        raise ValueError("a query sees no key")
    s = (np.asarray(q, np.float64) @ K.T) * sm_scale
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.where(visible, np.exp(s - m), 0.0)
    p = e / e.sum(axis=1, keepdims=True)
    return p @ V


def head_slice(B: np.ndarray, h: int, head_dim: int) -> np.ndarray:
    """Columns [hD, (h+1)D) of an adapter matrix [r, Hkv*D]."""
    return np.asarray(B, np.float64)[:, h * head_dim:(h + 1) * head_dim]


def residual_attention(q: np.ndarray, q_positions: np.ndarray,
                       k_base: np.ndarray, v_base: np.ndarray,
                       k_res: np.ndarray, v_res: np.ndarray,
                       B_k: np.ndarray, B_v: np.ndarray,
                       theta: float, sm_scale: Optional[float] = None,
                       key_positions: Optional[np.ndarray] = None,
                       seq_len: Optional[int] = None,
                       q_heads: Optional[Sequence[int]] = None) -> np.ndarray:
    """ResidualAttention of ONE agent against its disaggregated cache (fp64).

    q [Nq, Hq, D] (already rotated), q_positions [Nq];
    k_base, v_base [L, Hkv, D] (base rows, keys already rotated);
    k_res, v_res [L, r] (residual rows, unrotated); B_k, B_v [r, Hkv*D].
    Keys j < seq_len (default L) with key_positions[j] <= q_positions[t] are
    visible to query t.  Returns O [Nq, Hq, D]; heads not in ``q_heads`` are NaN.
    """
    q = np.asarray(q, np.float64)
    Nq, Hq, D = q.shape
    L, Hkv, _ = k_base.shape
    if seq_len is None:
        seq_len = L
    if key_positions is None:
        key_positions = np.arange(L, dtype=np.int64)
    key_positions = np.asarray(key_positions)[:seq_len]
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    G = Hq // Hkv
    visible = key_positions[None, :] <= np.asarray(q_positions)[:, None]
    heads = range(Hq) if q_heads is None else q_heads
    out = np.full((Nq, Hq, D), np.nan)
    for h in sorted({hq // G for hq in heads}):
        K = residual_keys(np.asarray(k_base[:seq_len, h]), k_res[:seq_len], head_slice(B_k, h, D),
                          key_positions, theta)
        V = residual_values(np.asarray(v_base[:seq_len, h]), v_res[:seq_len], head_slice(B_v, h, D))
        for hq in heads:
            if hq // G == h:
                out[:, hq] = softmax_attention(q[:, hq], K, V, visible, sm_scale)
    return out


def residual_attention_online(q_vec: np.ndarray, q_position: int,
                              k_base_h: np.ndarray, v_base_h: np.ndarray,
                              k_res: np.ndarray, v_res: np.ndarray,
                              B_k_h: np.ndarray, B_v_h: np.ndarray,
                              theta: float, sm_scale: float, block: int = 16) -> np.ndarray:
    """The kernel's order of work, in fp64, for one query vector and one KV head.

    Restates ForkKV L2 section 7 (implementation cross-reference) and section 4
    check 6: keys are visited block by block; each block's residual keys are
    up-projected and rotated at their positions, added to the base keys, and
    scored; a running maximum m and normaliser l are kept, and BOTH the base
    accumulator acc (D wide) and the residual accumulator acc_r (r wide) are
    rescaled by exp(m - m_new) when m grows.  B_v is applied once at the end:
    out = (acc + acc_r B_v) / l.
    """
    L = k_base_h.shape[0]
    D = k_base_h.shape[1]
    r = k_res.shape[1]
    m, l = -np.inf, 0.0
    acc = np.zeros(D)
    acc_r = np.zeros(r)
    q_vec = np.asarray(q_vec, np.float64)
    for j0 in range(0, L, block):
        j1 = min(L, j0 + block)
        pos = np.arange(j0, j1)
        vis = pos <= q_position
        if not vis.any():
            continue
        K = residual_keys(k_base_h[j0:j1], k_res[j0:j1], B_k_h, pos, theta)
        s = np.where(vis, (K @ q_vec) * sm_scale, -np.inf)
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m > -np.inf else 0.0
        p = np.where(vis, np.exp(s - m_new), 0.0)
        l = alpha * l + p.sum()
        acc = alpha * acc + p @ np.asarray(v_base_h[j0:j1], np.float64)
        acc_r = alpha * acc_r + p @ np.asarray(v_res[j0:j1], np.float64)
        m = m_new
    return (acc + acc_r @ np.asarray(B_v_h, np.float64)) / l


def metrics(out: np.ndarray, ref: np.ndarray) -> dict:
    """Max-abs and relative-L2 error of ``out`` against ``ref`` (finite entries of ref)."""
    mask = np.isfinite(ref)
    d = np.asarray(out, np.float64)[mask] - ref[mask]
    rn = float(np.linalg.norm(ref[mask]))
    return {"max_abs": float(np.abs(d).max()) if d.size else 0.0,
            "rel_l2": float(np.linalg.norm(d) / rn) if rn > 0 else float(np.linalg.norm(d))}


# Tolerance stated with the method's target: bf16 inputs, fp32 accumulation.
TOL_MAX_ABS = 2e-2
TOL_REL_L2 = 5e-3


def within_tolerance(out: np.ndarray, ref: np.ndarray) -> bool:
    e = metrics(out, ref)
    return e["max_abs"] <= TOL_MAX_ABS and e["rel_l2"] <= TOL_REL_L2
