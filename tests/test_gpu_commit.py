"""LCP commit end to end on the GPU (ForkServe README, "Methods": bind the observed
token prefix, CoW-split a mid-page, abort the siblings; decode then uses only KV
that matches the committed sequence).

A 40-token trunk forks two speculative branches that each append 30 tokens.
The observed tokens agree with branch 1 for the first 20 tokens only, inside the
trunk's second page, which the trunk still uses: the commit aborts branch 2,
truncates branch 1 and splits that page (a copy of its first 4 rows).  Branch 1
then appends 6 observed tokens into its private copy.  Decode of branch 1 and of
the trunk must both match the fp64 oracle on their own logical sequences, which
they only can if the split copied the committed rows and left the trunk's page
untouched.
"""
import numpy as np
import pytest
import torch

from gpu_harness import record

from disaggregated_kv_attention_gb300 import forkkv as fk
from disaggregated_kv_attention_gb300.paged import _slots
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
    kb = torch.randn(n, HKV, D, generator=g).to(torch.bfloat16)
    vb = torch.randn(n, HKV, D, generator=g).to(torch.bfloat16)
    kr = torch.randn(n, R, generator=g).to(torch.bfloat16)
    vr = torch.randn(n, R, generator=g).to(torch.bfloat16)
    return kb, vb, kr, vr


def _write(pools, alloc, seq, start, rows, base=True):
    """Rows for logical positions [start, start + n) of seq (base rows only if base)."""
    kb, vb, kr, vr = rows
    n = kr.shape[0]
    npg = (start + n + 15) // 16
    b, r, _ = fk.forkkv_page_tables(alloc, [seq], npg)
    sb = torch.from_numpy(_slots(b[0], start, n)).cuda()
    sr = torch.from_numpy(_slots(r[0], start, n)).cuda()
    if base:
        fk.forkkv_write_rows(pools, 0, sb, sr, kb.cuda(), vb.cuda(), kr.cuda(), vr.cuda())
    else:
        fk.forkkv_write_rows(pools, 0, None, sr, None, None, kr.cuda(), vr.cuda())


@pytest.mark.parametrize("use_plan", [False, True])
def test_commit_split_then_decode_matches_oracle(use_plan):
    g = torch.Generator().manual_seed(31)
    alloc = fk.forkkv_alloc_create(64, 64)
    pools = fk.Pools(64, 64, HKV, n_layers=1, fill=0)
    trunk = _rows(g, 40)
    T = fk.forkkv_seq_create(alloc, 40)
    _write(pools, alloc, T, 0, trunk)
    b1, j1 = fk.forkkv_fork(alloc, T, 40)
    b2, j2 = fk.forkkv_fork(alloc, T, 40)
    fk.forkkv_cow_copy_rows(pools, j1 + j2)  # the 8-row tail of the trunk, packed into each branch
    res_prefix = {}
    spec = {}
    for b in (b1, b2):
        res_prefix[b] = _rows(g, 40)
        _write(pools, alloc, b, 0, res_prefix[b], base=False)  # the branch's own xA rows of the prefix
        assert fk.forkkv_append(alloc, b, 30) == []
        spec[b] = _rows(g, 30)
        _write(pools, alloc, b, 40, spec[b])
    trunk_tokens = list(range(100, 140))
    b1_tokens = trunk_tokens + list(range(500, 530))
    observed = trunk_tokens[:20] + [7] * 10  # diverges from the trunk itself at token 20
    lcp = fk.forkkv_lcp_len(b1_tokens, observed)
    assert lcp == 20
    b1_pages_before = fk.forkkv_page_tables(alloc, [b1], 5)[0][0]
    jobs = fk.forkkv_commit(alloc, b1, lcp, [b2])
    assert len(jobs) == 1 and jobs[0][0] == b1_pages_before[1] and jobs[0][2] == 4 and jobs[0][3] == fk.JOB_BASE
    fk.forkkv_cow_copy_rows(pools, jobs)
    assert fk.forkkv_append(alloc, b1, 6) == []  # the split page is private now
    new = _rows(g, 6)
    _write(pools, alloc, b1, 20, new)

    # decode: branch 1 (26 tokens) and the trunk (40 tokens), one query token each
    agents = [b1, T]
    lens = [26, 40]
    stride = 3
    bpt, rpt, sl = fk.forkkv_page_tables(alloc, agents, stride)
    assert list(sl) == lens
    q = torch.randn(2, 1, HKV * G, D, generator=g).to(torch.bfloat16)
    B_k = (0.2 * torch.randn(2, R, HKV * D, generator=g)).to(torch.bfloat16)
    B_v = (0.2 * torch.randn(2, R, HKV * D, generator=g)).to(torch.bfloat16)
    dev = torch.device("cuda", 0)
    qd, out = q.to(dev), torch.empty(2, 1, HKV * G, D, dtype=torch.bfloat16, device=dev)
    bpt_t, rpt_t = torch.from_numpy(bpt).to(dev), torch.from_numpy(rpt).to(dev)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=dev)
    pos_t = torch.tensor([[25], [39]], dtype=torch.int32, device=dev)
    Bk_d, Bv_d = B_k.to(dev), B_v.to(dev)
    rope = fk.rope_table(THETA, 40, device=dev)
    plan_t, info = None, None
    if use_plan:
        plan, info = fk.forkkv_plan_build(bpt, np.array(lens, np.int32), HKV)
        plan_t = torch.from_numpy(plan).to(dev)
    p = fk.attn_params(pools, 0, qd, out, bpt_t, rpt_t, lens_t, pos_t, 40, Bk_d, Bv_d, rope=rope,
                       rope_theta=THETA, plan=plan_t, plan_info=info)
    ws = fk.workspace_for(p, prefill=False, device=dev)
    fk.forkkv_residual_attn_decode(p)
    torch.cuda.synchronize()
    assert fk.forkkv_get_device_status() == 0
    del ws

    def f64(t):
        return t.to(torch.float64).numpy()

    # logical sequences: branch 1 = trunk rows 0..19 + the 6 new rows; its residual rows are its own
    seqs = {
        0: (torch.cat([trunk[0][:20], new[0]]), torch.cat([trunk[1][:20], new[1]]),
            torch.cat([res_prefix[b1][2][:20], new[2]]), torch.cat([res_prefix[b1][3][:20], new[3]])),
        1: trunk,
    }
    got = out.to(torch.float64).cpu().numpy()
    for i, (kb, vb, kr, vr) in seqs.items():
        ref = ra.residual_attention(f64(q[i]), np.array([lens[i] - 1]), f64(kb), f64(vb), f64(kr), f64(vr),
                                    f64(B_k[i]), f64(B_v[i]), THETA)
        m = ra.metrics(got[i], ref)
        record(m)
        assert ra.within_tolerance(got[i], ref), (i, m)
    fk.forkkv_alloc_destroy(alloc)
