"""Freeze-tail forks on the GPU (ForkServe README, adaptive unaligned tail: one
read-only tail page shared by the children; "freeze-tail needs a fork-aware slot
map").

A 40-token trunk (its last page holds 8 rows) forks three children with
FORKKV_FORK_FREEZE_TAIL: no row is copied, each child's slots 40..47 are a hole
and its own tokens start on a fresh page, while the trunk writes its next tokens
into the shared page in place.  The pools start filled with NaN bit patterns, so
a hidden or never-written row that reached the value products would show.  Decode
of the children and the trunk, and a causal prefill chunk of a child, must match
the fp64 oracle on each agent's logical sequence (tokens at positions 0, 1, ...).
"""
import numpy as np
import pytest
import torch

from gpu_harness import record

from disaggregated_kv_attention_gb300 import forkkv as fk
from disaggregated_kv_attention_gb300.paged import token_slots
from oracle import residual_attention as ra

pytestmark = pytest.mark.gpu

HKV, G, D, R = 2, 4, 128, 16
THETA = 500000.0


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    fk.lib()
    assert fk.forkkv_get_device_status() == 0


def _rows(g, n):
    return (torch.randn(n, HKV, D, generator=g).to(torch.bfloat16), torch.randn(n, HKV, D, generator=g).to(torch.bfloat16),
            torch.randn(n, R, generator=g).to(torch.bfloat16), torch.randn(n, R, generator=g).to(torch.bfloat16))


def _write(pools, alloc, seq, start, rows, base=True):
    """Rows of tokens [start, start + n) of seq, through its slot map."""
    kb, vb, kr, vr = rows
    n = kr.shape[0]
    hole = fk.forkkv_slot_maps(alloc, [seq])[0]
    slots = token_slots(hole, start, n)
    b, r, _ = fk.forkkv_page_tables(alloc, [seq], int(slots.max()) // 16 + 1)
    sb = torch.from_numpy((b[0][slots // 16].astype(np.int64) * 16 + slots % 16).astype(np.int32)).cuda()
    sr = torch.from_numpy((r[0][slots // 16].astype(np.int64) * 16 + slots % 16).astype(np.int32)).cuda()
    if base:
        fk.forkkv_write_rows(pools, 0, sb, sr, kb.cuda(), vb.cuda(), kr.cuda(), vr.cuda())
    else:
        fk.forkkv_write_rows(pools, 0, None, sr, None, None, kr.cuda(), vr.cuda())


def _cat(*parts):
    return tuple(torch.cat([p[i] for p in parts]) for i in range(4))


def _tree(g):
    alloc = fk.forkkv_alloc_create(64, 64)
    pools = fk.Pools(64, 64, HKV, n_layers=1, fill=0xFF)  # 0xFFFF: a NaN in every unwritten bf16
    trunk = _rows(g, 40)
    T = fk.forkkv_seq_create(alloc, 40)
    _write(pools, alloc, T, 0, trunk)
    kids, logical = [], {}
    for i, own in enumerate((20, 5, 33)):
        c, jobs = fk.forkkv_fork(alloc, T, 40, fk.FORK_FREEZE_TAIL)
        assert all(j[3] in (fk.JOB_BASE_ZERO, fk.JOB_RES_ZERO) for j in jobs) and len(jobs) == 2
        fk.forkkv_cow_copy_rows(pools, jobs)          # zero the shared page's empty rows first
        assert tuple(fk.forkkv_slot_maps(alloc, [c])[0]) == (40, 8)
        prefix_res = _rows(g, 40)
        _write(pools, alloc, c, 0, prefix_res, base=False)
        assert fk.forkkv_append(alloc, c, own) == []
        mine = _rows(g, own)
        _write(pools, alloc, c, 40, mine)
        kids.append(c)
        logical[c] = _cat(trunk[:2] + prefix_res[2:], mine)
        if i == 0:
            # the trunk writes on into its frozen tail in place (the children read rows 0..7 only)
            assert fk.forkkv_append(alloc, T, 6) == []
            more = _rows(g, 6)
            _write(pools, alloc, T, 40, more)
            logical[T] = _cat(trunk, more)
    return alloc, pools, kids, T, logical


def _f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("use_plan", [False, True])
def test_freeze_decode_matches_oracle(use_plan):
    g = torch.Generator().manual_seed(41)
    alloc, pools, kids, T, logical = _tree(g)
    agents = kids + [T]
    A = len(agents)
    bpt, rpt, slots = fk.forkkv_page_tables(alloc, agents, 8)
    holes = fk.forkkv_slot_maps(alloc, agents)
    lens = [fk.forkkv_seq_len(alloc, s) for s in agents]
    assert list(slots) == [l + int(h[1]) for l, h in zip(lens, holes)]
    dev = torch.device("cuda", 0)
    q = torch.randn(A, 1, HKV * G, D, generator=g).to(torch.bfloat16)
    B_k = (0.2 * torch.randn(A, R, HKV * D, generator=g)).to(torch.bfloat16)
    B_v = (0.2 * torch.randn(A, R, HKV * D, generator=g)).to(torch.bfloat16)
    out = torch.empty(A, 1, HKV * G, D, dtype=torch.bfloat16, device=dev)
    pos = torch.tensor([[l - 1] for l in lens], dtype=torch.int32, device=dev)
    max_len = int(max(slots))
    rope = fk.rope_table(THETA, max_len, device=dev)
    plan_t, info = None, None
    if use_plan:
        plan, info = fk.forkkv_plan_build(bpt, slots.astype(np.int32), HKV)
        plan_t = torch.from_numpy(plan).to(dev)
        assert info.n_items < A * 2  # the trunk pages are one shared item
    qd = q.to(dev)
    tensors = [torch.from_numpy(x).to(dev) for x in (bpt, rpt, slots.astype(np.int32), holes)]
    Bk_d, Bv_d = B_k.to(dev), B_v.to(dev)
    p = fk.attn_params(pools, 0, qd, out, tensors[0], tensors[1], tensors[2], pos, max_len, Bk_d, Bv_d, rope=rope,
                       rope_theta=THETA, plan=plan_t, plan_info=info, holes=tensors[3])
    ws = fk.workspace_for(p, prefill=False, device=dev)
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    del ws
    got = out.to(torch.float64).cpu().numpy()
    for i, s in enumerate(agents):
        kb, vb, kr, vr = logical[s]
        assert kb.shape[0] == lens[i]
        ref = ra.residual_attention(_f64(q[i]), np.array([lens[i] - 1]), _f64(kb), _f64(vb), _f64(kr), _f64(vr),
                                    _f64(B_k[i]), _f64(B_v[i]), THETA)
        record(ra.metrics(got[i], ref))
        assert ra.within_tolerance(got[i], ref), (i, ra.metrics(got[i], ref))
    fk.forkkv_alloc_destroy(alloc)


def test_freeze_prefill_chunk_matches_oracle():
    """A child forked with a frozen tail prefills a causal 300-token chunk after its hole."""
    g = torch.Generator().manual_seed(43)
    alloc, pools, kids, T, logical = _tree(g)
    c = kids[1]                                    # 5 own tokens so far (slots 48..52)
    C = 300
    assert fk.forkkv_append(alloc, c, C) == []
    chunk = _rows(g, C)
    _write(pools, alloc, c, 45, chunk)
    kb, vb, kr, vr = _cat(logical[c], chunk)
    L = fk.forkkv_seq_len(alloc, c)
    assert L == 45 + C
    dev = torch.device("cuda", 0)
    bpt, rpt, slots = fk.forkkv_page_tables(alloc, [c], 32)
    holes = fk.forkkv_slot_maps(alloc, [c])
    q = torch.randn(1, C, HKV * G, D, generator=g).to(torch.bfloat16)
    B_k = (0.2 * torch.randn(1, R, HKV * D, generator=g)).to(torch.bfloat16)
    B_v = (0.2 * torch.randn(1, R, HKV * D, generator=g)).to(torch.bfloat16)
    positions = torch.arange(45, 45 + C, dtype=torch.int32).view(1, C)
    out = torch.empty(1, C, HKV * G, D, dtype=torch.bfloat16, device=dev)
    max_len = int(slots[0])
    rope = fk.rope_table(THETA, max_len, device=dev)
    tensors = [torch.from_numpy(x).to(dev) for x in (bpt, rpt, slots.astype(np.int32), holes)]
    p = fk.attn_params(pools, 0, q.to(dev), out, tensors[0], tensors[1], tensors[2], positions.to(dev), max_len,
                       B_k.to(dev), B_v.to(dev), rope=rope, rope_theta=THETA, holes=tensors[3])
    ws = fk.workspace_for(p, prefill=True, device=dev)
    fk.forkkv_residual_attn_prefill_chunk(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    del ws
    got = out[0].to(torch.float64).cpu().numpy()
    ref = ra.residual_attention(_f64(q[0]), positions[0].numpy(), _f64(kb), _f64(vb), _f64(kr), _f64(vr),
                                _f64(B_k[0]), _f64(B_v[0]), THETA)
    record(ra.metrics(got, ref))
    assert ra.within_tolerance(got, ref), ra.metrics(got, ref)
    fk.forkkv_alloc_destroy(alloc)
