"""Pins of the fp64 attention oracle against what the pages and mathematics fix.

Each test below would fail for a plausible mistake in the oracle: a dropped
residual term, a wrong RoPE pairing or angle, a wrong head slice of B, a wrong
softmax scale, an off-by-one mask, or an un-rescaled residual accumulator.
"""
import math

import numpy as np
import pytest
import torch

from oracle import residual_attention as ra
from disaggregated_kv_attention_gb300 import workload as wl


def _np(t):
    return t.to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# Hand-derived tiny cases (brute force by hand; pure closed forms)
# ---------------------------------------------------------------------------

def _one_agent(q, qpos, kb, vb, kr, vr, Bk, Bv, theta=10000.0):
    # shapes: q [Nq, D] (one head), kb/vb [L, D], kr/vr [L, r], B [r, D]
    q = np.asarray(q, float)[:, None, :]
    kb = np.asarray(kb, float)[:, None, :]
    vb = np.asarray(vb, float)[:, None, :]
    return ra.residual_attention(q, np.asarray(qpos), kb, vb, np.asarray(kr, float), np.asarray(vr, float),
                                 np.asarray(Bk, float), np.asarray(Bv, float), theta)[:, 0, :]


def test_single_key_returns_value_exactly():
    # D=2, r=1, one key at position 0: softmax weight 1, O = Vb + Vr*B_v = [1 + 3*0.5, 2 - 3].
    out = _one_agent([[1.0, 1.0]], [0], [[0.5, -1.0]], [[1.0, 2.0]], [[3.0]], [[3.0]], [[1.0, 1.0]], [[0.5, -1.0]])
    assert np.allclose(out, [[2.5, -1.0]], atol=1e-15, rtol=0)


def _case_b():
    # D=2, r=1, query at position 1 with scale 1/sqrt(2) and q=[sqrt2, 0] so s_j = K_j[0].
    # key 0: Kb=[-2,0], Kr=2, B_k=[1,0] -> U=[2,0], RoPE at 0 is the identity -> K=[0,0], s0=0.
    # key 1: Kr=1 -> U=[1,0], RoPE by 1 rad -> [cos1, sin1]; Kb=[ln3 - cos1, 0] -> s1 = ln 3.
    # weights (1/4, 3/4); V0 = [4,0]; V1 = Vb + Vr*B_v = [0,2] + 2*[0,1] = [0,4] -> O = [1, 3].
    ln3, c1 = math.log(3.0), math.cos(1.0)
    kb = [[-2.0, 0.0], [ln3 - c1, 0.0]]
    vb = [[4.0, 0.0], [0.0, 2.0]]
    kr = [[2.0], [1.0]]
    vr = [[0.0], [2.0]]
    return kb, vb, kr, vr, [[1.0, 0.0]], [[0.0, 1.0]]


def test_two_keys_deferred_rope_and_value_residual():
    kb, vb, kr, vr, Bk, Bv = _case_b()
    out = _one_agent([[math.sqrt(2.0), 0.0]], [1], kb, vb, kr, vr, Bk, Bv)
    assert np.allclose(out, [[1.0, 3.0]], atol=1e-14, rtol=0)


def test_mask_hides_future_keys():
    # case B plus a third key at position 2 whose score would dominate; the query sits at 1.
    kb, vb, kr, vr, Bk, Bv = _case_b()
    kb = kb + [[100.0, 0.0]]
    vb = vb + [[1000.0, 1000.0]]
    kr = kr + [[0.0]]
    vr = vr + [[0.0]]
    out = _one_agent([[math.sqrt(2.0), 0.0]], [1], kb, vb, kr, vr, Bk, Bv)
    assert np.allclose(out, [[1.0, 3.0]], atol=1e-14, rtol=0)


def test_causal_chunk_two_queries():
    # queries at positions 0 and 1 over case B's keys: the first sees only key 0 -> V0 = [4, 0].
    kb, vb, kr, vr, Bk, Bv = _case_b()
    s2 = math.sqrt(2.0)
    out = _one_agent([[s2, 0.0], [s2, 0.0]], [0, 1], kb, vb, kr, vr, Bk, Bv)
    assert np.allclose(out, [[4.0, 0.0], [1.0, 3.0]], atol=1e-14, rtol=0)


def test_rotate_half_pairing_d4():
    # D=4, theta=1e4: frequencies (1, 0.01).  U=[0,0,1,0] at position 1: rotate-half pairs (0,2)
    # -> [-sin1, 0, cos1, 0]; an interleaved pairing would leave component 0 at 0.
    # Kb1 = [ln3 + sin1, 0, 0, 0] makes s1 = ln 3 (scale 1/2, q = [2,0,0,0]); O = [1, 3, 0, 0].
    ln3, s1 = math.log(3.0), math.sin(1.0)
    kb = [[0, 0, 0, 0], [ln3 + s1, 0, 0, 0]]
    vb = [[4, 0, 0, 0], [0, 4, 0, 0]]
    out = _one_agent([[2.0, 0, 0, 0]], [1], kb, vb, [[0.0], [1.0]], [[0.0], [0.0]],
                     [[0, 0, 1.0, 0]], [[0, 0, 0, 0.0]])
    assert np.allclose(out, [[1.0, 3.0, 0.0, 0.0]], atol=1e-14, rtol=0)


@pytest.mark.parametrize("i", [0, 1, 2, 3])
def test_rope_frequency_of_every_pair_index_d8(i):
    # D=8, theta=1e4: the angular frequency of pair index i is 1e4^(-2i/8) = 10^-i exactly, so a
    # key at position 10^i is turned by exactly 1 rad on pair (i, i+4) and by 10^(i-k) rad on the
    # others.  A unit vector on component i+4 must come out as -sin 1 on i and cos 1 on i+4
    # (written out by hand: (a, b) -> (a cos - b sin, b cos + a sin) with a=0, b=1).  A wrong
    # exponent (theta^(-i/D), a D-2 denominator, 0-based vs 1-based pair index) moves the angle.
    x = np.zeros((1, 8))
    x[0, i + 4] = 1.0
    got = ra.rope_rotate_half(x, np.array([10 ** i]), 1e4)[0]
    want = np.zeros(8)
    want[i], want[i + 4] = -math.sin(1.0), math.cos(1.0)
    assert np.allclose(got, want, atol=1e-12, rtol=0)


def test_rope_second_frequency_through_attention_d4():
    # D=4, theta=1e4: pair index 1 has frequency 1e4^(-2/4) = 0.01 exactly.  Keys sit at
    # positions 0 and 100 (key_positions), the query at 100.  Key 1: U = 1*[0,0,0,1]; pair (1,3)
    # turned by 100*0.01 = 1 rad -> K_lora = [0, -sin1, 0, cos1].  With q = [0,-2,0,0], scale 1/2
    # and Kb1 = [0, sin1 - ln3, 0, 0]: s1 = -(sin1 - ln3 - sin1) = ln 3; key 0 scores 0.
    # Weights (1/4, 3/4), V0 = [4,0,0,0], V1 = [0,4,0,0] -> O = [1, 3, 0, 0].
    ln3, s1 = math.log(3.0), math.sin(1.0)
    q = np.array([[[0.0, -2.0, 0.0, 0.0]]])
    kb = np.array([[[0.0, 0, 0, 0]], [[0.0, s1 - ln3, 0, 0]]])
    vb = np.array([[[4.0, 0, 0, 0]], [[0.0, 4, 0, 0]]])
    out = ra.residual_attention(q, np.array([100]), kb, vb, np.array([[0.0], [1.0]]), np.zeros((2, 1)),
                                np.array([[0.0, 0, 0, 1]]), np.zeros((1, 4)), 1e4,
                                key_positions=np.array([0, 100]))
    assert np.allclose(out[:, 0, :], [[1.0, 3.0, 0.0, 0.0]], atol=1e-14, rtol=0)


def test_hand_cases_through_online_restatement():
    kb, vb, kr, vr, Bk, Bv = _case_b()
    for block in (1, 2):
        out = ra.residual_attention_online(np.array([math.sqrt(2.0), 0.0]), 1, np.array(kb), np.array(vb),
                                           np.array(kr), np.array(vr), np.array(Bk), np.array(Bv),
                                           10000.0, 1.0 / math.sqrt(2.0), block=block)
        assert np.allclose(out, [1.0, 3.0], atol=1e-14, rtol=0)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("p", [0, 1, 2 ** 17])
def test_rope_is_complex_rotation(p):
    rng = np.random.default_rng(3)
    D, theta = 128, 500000.0
    x = rng.standard_normal((1, D))
    z = x[0, :D // 2] + 1j * x[0, D // 2:]
    f = theta ** (-np.arange(0, D, 2, dtype=np.float64) / D)
    zr = z * np.exp(1j * p * f)
    want = np.concatenate([zr.real, zr.imag])
    got = ra.rope_rotate_half(x, np.array([p]), theta)[0]
    assert np.allclose(got, want, atol=1e-12, rtol=0)
    if p == 0:
        assert np.array_equal(got, x[0])


def test_rope_relative_shift_invariance():
    # Rotating q and every key by the same extra offset leaves all scores, hence O, unchanged.
    rng = np.random.default_rng(4)
    L, Hkv, G, D, r, theta = 37, 2, 3, 128, 16, 1e6
    q_raw = rng.standard_normal((1, Hkv * G, D))
    kb_raw = rng.standard_normal((L, Hkv, D))
    vb = rng.standard_normal((L, Hkv, D))
    kr, vr = rng.standard_normal((L, r)), rng.standard_normal((L, r))
    Bk, Bv = 0.1 * rng.standard_normal((r, Hkv * D)), 0.1 * rng.standard_normal((r, Hkv * D))
    outs = []
    for delta in (0, 1000, 77777):
        kp = np.arange(L) + delta
        qp = np.array([L - 1 + delta])
        kb = np.stack([ra.rope_rotate_half(kb_raw[:, h], kp, theta) for h in range(Hkv)], axis=1)
        q = np.stack([ra.rope_rotate_half(q_raw[:, hq], qp, theta) for hq in range(Hkv * G)], axis=1)
        outs.append(ra.residual_attention(q, qp, kb, vb, kr, vr, Bk, Bv, theta, key_positions=kp))
    assert np.allclose(outs[0], outs[1], atol=1e-9, rtol=0)
    assert np.allclose(outs[0], outs[2], atol=1e-9, rtol=0)


# ---------------------------------------------------------------------------
# Special cases reducing to a library routine or a closed form
# ---------------------------------------------------------------------------

def _sdpa_gqa(q, k, v, mask):
    # q [Nq, Hq, D]; k, v [L, Hkv, D]; mask [Nq, L] bool -> torch fp64 SDPA with repeated KV heads
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.from_numpy(mask))
    return o.permute(1, 0, 2).numpy()


@pytest.mark.parametrize("cfg_name", ["tiny_decode"])
def test_zero_adapters_reduce_to_plain_gqa(cfg_name):
    w = wl.generate(wl.CONFIGS[cfg_name])
    for a in range(w.n_agents):
        kb, vb = w.agent_base(a)
        L = kb.shape[0]
        zeros = np.zeros((16, w.cfg.n_kv_heads * 128))
        out = ra.residual_attention(_np(w.q[a]), w.positions[a].numpy(), _np(kb), _np(vb),
                                    _np(w.k_res[a]), _np(w.v_res[a]), zeros, zeros, w.cfg.rope_theta)
        mask = np.arange(L)[None, :] <= w.positions[a].numpy()[:, None]
        ref = _sdpa_gqa(_np(w.q[a]), _np(kb), _np(vb), mask)
        assert np.allclose(out, ref, atol=1e-12, rtol=0)


def test_zero_adapters_causal_chunk_plain_gqa():
    rng = np.random.default_rng(5)
    L, C, Hkv, G, D = 50, 13, 2, 5, 128
    q = rng.standard_normal((C, Hkv * G, D))
    kb, vb = rng.standard_normal((L, Hkv, D)), rng.standard_normal((L, Hkv, D))
    qp = np.arange(L - C, L)
    z = np.zeros((16, Hkv * D))
    out = ra.residual_attention(q, qp, kb, vb, rng.standard_normal((L, 16)), rng.standard_normal((L, 16)), z, z, 1e6)
    ref = _sdpa_gqa(q, kb, vb, np.arange(L)[None, :] <= qp[:, None])
    assert np.allclose(out, ref, atol=1e-12, rtol=0)


def test_zero_query_gives_mean_value():
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    a = 1
    kb, vb = w.agent_base(a)
    q = np.zeros_like(_np(w.q[a]))
    out = ra.residual_attention(q, w.positions[a].numpy(), _np(kb), _np(vb), _np(w.k_res[a]),
                                _np(w.v_res[a]), _np(w.B_k[a]), _np(w.B_v[a]), w.cfg.rope_theta)
    # uniform weights: O = mean(Vb) + mean(Vr) @ B_v, with the means taken first.
    G = w.cfg.group
    for hq in range(w.cfg.n_q_heads):
        h = hq // G
        want = _np(vb)[:, h].mean(0) + _np(w.v_res[a]).mean(0) @ _np(w.B_v[a])[:, h * 128:(h + 1) * 128]
        assert np.allclose(out[0, hq], want, atol=1e-12, rtol=0)


def test_disaggregated_equals_merged_by_linearity():
    # bCache = RoPE(x W_k), rCache = x A_k; merged cache = RoPE(x (W_k + A_k B_k)).
    rng = np.random.default_rng(6)
    L, hidden, Hkv, D, r, theta = 40, 96, 2, 128, 16, 5e5
    x = rng.standard_normal((L, hidden))
    Wk, Wv = rng.standard_normal((hidden, Hkv * D)), rng.standard_normal((hidden, Hkv * D))
    Ak, Av = 0.02 * rng.standard_normal((hidden, r)), 0.02 * rng.standard_normal((hidden, r))
    Bk, Bv = 0.02 * rng.standard_normal((r, Hkv * D)), 0.02 * rng.standard_normal((r, Hkv * D))
    pos = np.arange(L)
    kb = np.stack([ra.rope_rotate_half((x @ Wk)[:, h * D:(h + 1) * D], pos, theta) for h in range(Hkv)], 1)
    vb = (x @ Wv).reshape(L, Hkv, D)
    kr, vr = x @ Ak, x @ Av
    Wk_m, Wv_m = Wk + Ak @ Bk, Wv + Av @ Bv
    for h in range(Hkv):
        merged_k = ra.rope_rotate_half((x @ Wk_m)[:, h * D:(h + 1) * D], pos, theta)
        merged_v = (x @ Wv_m)[:, h * D:(h + 1) * D]
        got_k = ra.residual_keys(kb[:, h], kr, ra.head_slice(Bk, h, D), pos, theta)
        got_v = ra.residual_values(vb[:, h], vr, ra.head_slice(Bv, h, D))
        assert np.allclose(got_k, merged_k, atol=1e-12 * np.abs(merged_k).max(), rtol=0)
        assert np.allclose(got_v, merged_v, atol=1e-12 * np.abs(merged_v).max(), rtol=0)
    # and the attention over the merged cache, through torch SDPA
    q = rng.standard_normal((1, Hkv * 4, D))
    qp = np.array([L - 1])
    out = ra.residual_attention(q, qp, kb, vb, kr, vr, Bk, Bv, theta)
    km = np.stack([ra.rope_rotate_half((x @ Wk_m)[:, h * D:(h + 1) * D], pos, theta) for h in range(Hkv)], 1)
    vm = (x @ Wv_m).reshape(L, Hkv, D)
    ref = _sdpa_gqa(q, km, vm, np.ones((1, L), bool))
    assert np.allclose(out, ref, atol=1e-10, rtol=0)


def test_online_restatement_equals_materialised_two_pass():
    # Associativity of the value path and the dual-accumulator rescale: the kernel's order of
    # work (acc + acc_r B_v at the end) reproduces the materialised softmax(QK^T) V.
    w = wl.generate(wl.CONFIGS["tiny_decode"])
    D = 128
    for a in range(w.n_agents):
        kb, vb = w.agent_base(a)
        ref = ra.residual_attention(_np(w.q[a]), w.positions[a].numpy(), _np(kb), _np(vb), _np(w.k_res[a]),
                                    _np(w.v_res[a]), _np(w.B_k[a]), _np(w.B_v[a]), w.cfg.rope_theta)
        for hq in (0, 5, 31):
            h = hq // w.cfg.group
            got = ra.residual_attention_online(_np(w.q[a, 0, hq]), int(w.positions[a, 0]), _np(kb[:, h]),
                                               _np(vb[:, h]), _np(w.k_res[a]), _np(w.v_res[a]),
                                               ra.head_slice(_np(w.B_k[a]), h, D),
                                               ra.head_slice(_np(w.B_v[a]), h, D),
                                               w.cfg.rope_theta, 1 / math.sqrt(D), block=16 + 7 * a)
            assert np.allclose(got, ref[0, hq], atol=1e-12, rtol=0)


def test_metrics_and_tolerance_constants():
    ref = np.array([3.0, 4.0])
    e = ra.metrics(np.array([3.0, 4.1]), ref)
    assert math.isclose(e["max_abs"], 0.1, rel_tol=1e-12)
    assert math.isclose(e["rel_l2"], 0.1 / 5.0, rel_tol=1e-12)
    assert ra.TOL_MAX_ABS == 2e-2 and ra.TOL_REL_L2 == 5e-3
