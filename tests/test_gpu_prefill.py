"""Prefill-chunk parity: the CUDA path through the C-ABI against the fp64 oracle.

The chunk's own rows are written first (forkkv_write_rows, via the harness),
then attended causally.  The 14B-shaped chunk (8 agents x 2048 tokens on a
16384-token prefix) is checked on sampled query rows of sampled agents and
heads; small cases are checked on every output.  Tolerance as for decode.
"""
import pytest
import torch

from disaggregated_kv_attention_gb300 import forkkv as fk
from disaggregated_kv_attention_gb300 import workload as wl
from gpu_harness import compare, oracle, params, place

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    fk.forkkv_get_device_status()


def _run(P, rope=None):
    out = torch.full_like(P.q, float("nan"))
    p, keep = params(P, out, rope=rope, prefill=True)
    fk.forkkv_residual_attn_prefill_chunk(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    return out


def test_prefill_parity_qwen25_14b_sampled():
    w = wl.generate(wl.CONFIGS["qwen25_14b_prefill"])
    P = place(w)
    out = _run(P, rope=fk.rope_table(w.cfg.rope_theta, P.max_seq_len))
    assert torch.isfinite(out.float()).all()
    rows = list(range(0, 24)) + list(range(1000, 1013)) + list(range(2030, 2048))
    G = w.cfg.group
    heads = list(range(0, G)) + list(range(7 * G, 8 * G))
    ref = oracle(w, [0, 5], q_heads=heads, q_rows=rows)
    m, ok = compare(out, ref, q_rows=rows)
    assert ok, m


def _custom(name, Hq, Hkv, nodes, q_len, theta=1e6, b_std=0.02):
    cfg = wl.custom_config(name, Hq, Hkv, nodes, q_len=q_len, rope_theta=theta)
    return wl.generate(cfg, b_std=b_std)


@pytest.mark.parametrize("Hq,Hkv,prefix,chunk", [(40, 8, 300, 37), (32, 8, 0, 64), (8, 1, 16, 130), (64, 8, 1000, 200),
                                                 (28, 4, 77, 1)])
def test_prefill_small_cases_all_outputs(Hq, Hkv, prefix, chunk):
    nodes = []
    if prefix:
        nodes.append(wl.Node("root", -1, (prefix, prefix), False))
    nodes += [wl.Node(f"a{i}", 0 if prefix else -1, (chunk, chunk), True) for i in range(3)]
    w = _custom(f"pf{Hq}_{prefix}_{chunk}", Hq, Hkv, nodes, q_len=chunk, b_std=0.2)
    P = place(w)
    out = _run(P)
    m, ok = compare(out, oracle(w, range(w.n_agents)))
    assert ok, m


def test_prefill_first_token_sees_only_itself():
    # empty prefix: query 0 attends to key 0 alone, so O = Vb_0 + Vr_0 B_v exactly (up to bf16 output)
    nodes = [wl.Node("a0", -1, (20, 20), True)]
    w = _custom("first", 16, 4, nodes, q_len=20)
    P = place(w)
    out = _run(P)
    ref = oracle(w, [0], q_rows=[0])
    m, ok = compare(out, ref, q_rows=[0])
    assert ok and m["max_abs"] < 1e-2, m


@pytest.mark.parametrize("bad", ["negative", "past_end"])
def test_prefill_position_outside_the_sequence_sets_bad_arg(bad):
    # A query position must name a slot of its sequence (0 <= p < seq_len).  One out of range is
    # reported through the device status word (FORKKV_DEV_BAD_ARG); the kernel still finishes.
    nodes = [wl.Node("root", -1, (40, 40), False), wl.Node("a0", 0, (24, 24), True)]
    w = _custom("badpos", 16, 4, nodes, q_len=24)
    P = place(w)
    P.positions[0, 5] = -1 if bad == "negative" else int(w.seq_lens[0])
    out = torch.full_like(P.q, float("nan"))
    p, keep = params(P, out, prefill=True)
    fk.forkkv_residual_attn_prefill_chunk(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == fk.DEV_BAD_ARG
    assert fk.forkkv_get_device_status() == 0  # read and cleared; the context is still usable


@pytest.mark.parametrize("Hq,Hkv,prefix,chunk", [(40, 8, 300, 37), (64, 8, 1000, 200), (8, 1, 16, 130)])
def test_prefill_is_deterministic_across_calls(Hq, Hkv, prefix, chunk):
    # The kernel's order of work is fixed, so repeated calls on the same inputs give the same bits;
    # a hand-off between warps that reads a buffer before it is written may show up as calls that
    # differ (or as NaN).  Calls are interleaved with another workload so that shared and tensor
    # memory hold other data between them.
    nodes = ([wl.Node("root", -1, (prefix, prefix), False)] if prefix else []) + \
        [wl.Node(f"a{i}", 0 if prefix else -1, (chunk, chunk), True) for i in range(3)]
    w = _custom(f"det{Hq}_{prefix}_{chunk}", Hq, Hkv, nodes, q_len=chunk, b_std=0.2)
    P = place(w)
    other = place(_custom("det_other", 32, 8, [wl.Node("b0", -1, (700, 700), True)], q_len=700))
    first = _run(P)
    assert torch.isfinite(first.float()).all()
    for _ in range(4):
        _run(other)
        again = _run(P)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
