"""Pins of the allocator model and the accounting formulas.

Pinned against numbers the pages print (the ForkServe page-count table and the
ForkKV 16-agent memory example, fixtures under tests/golden/) and against
invariants any refcounted page allocator must keep.
"""
import csv
import json
import math
import os
import random

import pytest

from oracle import accounting as acc
from oracle.allocator import (AllocatorError, AllocatorModel, ERR_INVALID_ARG, ERR_OUT_OF_PAGES,
                              JOB_BASE, JOB_BASE_ZERO, JOB_RES, JOB_RES_ZERO, lcp_len)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P = 16


def _table():
    with open(os.path.join(GOLDEN, "forkserve_page_counts.tsv")) as f:
        rows = [l for l in f if not l.startswith("#")]
    return list(csv.DictReader(rows, delimiter="\t"))


SCENARIOS = _table()


def _fanout_model(L, k, ell):
    m = AllocatorModel(100000, 100000, P)
    parent = m.seq_create(L)
    children = []
    for _ in range(k):
        c, jobs = m.fork(parent, L)
        children.append((c, jobs))
        m.append(c, ell)
    return m, parent, children


@pytest.mark.parametrize("row", SCENARIOS, ids=[r["scenario"] for r in SCENARIOS])
def test_forkserve_table_closed_forms(row):
    L, k, ell = int(row["L"]), int(row["k"]), int(row["l"])
    apc, fs = int(row["apc_blk"]), int(row["fs_blk"])
    assert acc.pages_clone(L, k, ell, P) == apc
    assert acc.pages_fork_pack(L, k, ell, P) == fs
    assert round(100 * (1 - fs / apc), 1) == float(row["save_pct"])
    gib = lambda blocks: blocks * P * 128 * 1024 / 2 ** 30
    assert round(gib(apc), 2) == float(row["apc_gib"])
    assert round(gib(fs), 2) == float(row["fs_gib"])


@pytest.mark.parametrize("row", SCENARIOS, ids=[r["scenario"] for r in SCENARIOS])
def test_forkserve_table_by_simulation(row):
    L, k, ell = int(row["L"]), int(row["k"]), int(row["l"])
    m, parent, children = _fanout_model(L, k, ell)
    assert m.stats()["base_live"] == int(row["fs_blk"])
    # the unaligned tail is packed: one job per child, copying exactly L mod P rows
    for c, jobs in children:
        if L % P:
            assert len(jobs) == 1 and jobs[0][2] == L % P and jobs[0][3] == JOB_BASE
            assert jobs[0][0] == m.seqs[parent].base[L // P]
        else:
            assert jobs == []
    # freeing the parent must not drop the trunk the children still use
    trunk = list(m.seqs[parent].base[:L // P])
    m.free(parent)
    assert all(m.refcount(JOB_BASE, p) == k for p in trunk)
    # clone baseline: k independent sequences of L + l tokens
    c = AllocatorModel(100000, 100000, P)
    for _ in range(k):
        c.seq_create(L + ell)
    assert c.stats()["base_live"] == int(row["apc_blk"])


def test_pack_and_freeze_child_page_formulas():
    # unaligned_pack: L = 2050 (r = 2), k = 4, l = 48: pack = 4 * ceil(50/16) = 16; freeze = 1 + 4 * 3 = 13
    assert acc.pages_pack_children(2050, 4, 48, P) == 16
    assert acc.pages_freeze_children(2050, 4, 48, P) == 13
    # M_CoW vs M_clone with b = 1
    assert acc.m_cow(1, 2050, [48] * 4) == 2050 + 192
    assert acc.m_clone(1, 2050, [48] * 4) == 4 * 2050 + 192


def test_forkkv_memory_example():
    with open(os.path.join(GOLDEN, "forkkv_memory_example.json")) as f:
        ex = json.load(f)
    N, s, r, n = ex["n_agents"], ex["tokens"], ex["rank"], ex["width_n"]
    mdl = ex["model"]
    pr = ex["printed"]
    assert mdl["kv_heads"] * mdl["head_dim"] == n
    per_tok = acc.kv_bytes_per_token(mdl["layers"], mdl["kv_heads"], mdl["head_dim"], mdl["elem_bytes"])
    res_tok = acc.residual_bytes_per_token(mdl["layers"], r, mdl["elem_bytes"])
    unified = N * s * per_tok
    bcache = s * per_tok
    rcache = s * res_tok
    assert unified == pr["unified_gib"] * 2 ** 30
    assert bcache == pr["bcache_gib"] * 2 ** 30
    assert rcache == pr["rcache_mib_per_agent"] * 2 ** 20
    assert bcache // rcache == pr["size_ratio_n_over_r"] == n // r
    forkkv = bcache + N * rcache
    assert forkkv == pr["forkkv_gib_approx"] * 2 ** 30
    mr = acc.memory_ratio(N, r, n)
    assert mr == forkkv / unified == acc.memory_ratio_from_sizes(s, n, N, r) == 0.078125
    assert round(100 * r / n, 1) == pr["limit_ratio_percent_approx"]
    # the quoted 11.8x does not follow from the printed sizes; 64/5 = 12.8
    assert round(1 / mr, 1) == 12.8 and pr["quoted_reduction"] != 12.8


def test_memory_ratio_monotone():
    n = 1024
    for r in (8, 16, 64):
        vals = [acc.memory_ratio(N, r, n) for N in range(1, 65)]
        assert all(a > b for a, b in zip(vals, vals[1:]))
        assert abs(vals[-1] - (1 / 64 + r / n)) < 1e-15
    for N in (1, 4, 16):
        vals = [acc.memory_ratio(N, r, n) for r in (1, 2, 4, 8, 16, 32)]
        assert all(a < b for a, b in zip(vals, vals[1:]))


def test_memory_ratio_from_live_pages():
    # N agents forked from one s-token trunk: base pages counted once, residual pages per agent.
    s, N, r, n = 4096, 8, 16, 1024
    m = AllocatorModel(10000, 10000, P)
    root = m.seq_create(s)
    kids = [m.fork(root, s)[0] for _ in range(N)]
    m.free(root)
    st = m.stats()
    live = st["base_live"] * P * n + st["res_live"] * P * r
    assert live / (N * s * n) == acc.memory_ratio(N, r, n)


def _check_invariants(m: AllocatorModel):
    st = m.stats()
    base_refs = sum(len(s.base) for s in m.seqs.values())
    res_refs = sum(len(s.res) for s in m.seqs.values())
    assert st["base_refsum"] == base_refs and st["res_refsum"] == res_refs
    assert set(m.base_free).isdisjoint(p for s in m.seqs.values() for p in s.base)
    assert set(m.res_free).isdisjoint(p for s in m.seqs.values() for p in s.res)
    assert st["base_live"] + st["base_free"] == len(m.base_ref)
    assert st["res_live"] + st["res_free"] == len(m.res_ref)
    for s in m.seqs.values():
        assert len(s.base) == len(s.res) == math.ceil(s.slots() / P)
        assert s.hole_len == 0 or (0 < s.hole_len < P and (s.hole_start + s.hole_len) % P == 0)


def test_random_operations_keep_invariants():
    rnd = random.Random(7)
    m = AllocatorModel(300, 400, P)
    live = []
    for step in range(3000):
        op = rnd.random()
        snapshot = (list(m.base_free), list(m.res_free), list(m.base_ref), list(m.res_ref),
                    {k: (v.length, list(v.base), list(v.res)) for k, v in m.seqs.items()})
        try:
            if op < 0.2 or not live:
                live.append(m.seq_create(rnd.randint(0, 70)))
            elif op < 0.5:
                par = rnd.choice(live)
                c, _ = m.fork(par, rnd.randint(0, m.seqs[par].length), share_res=rnd.random() < 0.3,
                              freeze=rnd.random() < 0.4)
                live.append(c)
            elif op < 0.8:
                m.append(rnd.choice(live), rnd.randint(0, 40))
            else:
                sid = live.pop(rnd.randrange(len(live)))
                m.free(sid)
        except AllocatorError as e:
            assert e.code == ERR_OUT_OF_PAGES
            after = (m.base_free, m.res_free, m.base_ref, m.res_ref,
                     {k: (v.length, v.base, v.res) for k, v in m.seqs.items()})
            assert after == snapshot  # nothing changed on error
        _check_invariants(m)
    for sid in live:
        m.free(sid)
    assert m.stats()["base_free"] == 300 and m.stats()["res_free"] == 400
    assert sorted(m.base_free) == list(range(300))


def test_fork_share_res_and_append_cow():
    m = AllocatorModel(64, 64, P)
    root = m.seq_create(40)                      # pages 0,1,2 (last holds 8 rows)
    c, jobs = m.fork(root, 40, share_res=True)
    assert jobs == [(2, 3, 8, JOB_BASE), (2, 3, 8, JOB_RES)]
    assert m.seqs[c].base == [0, 1, 3] and m.seqs[c].res == [0, 1, 3]
    # a page-aligned fork aliases everything, then appending to a shared partial page copies it
    d, jobs = m.fork(root, 32)
    assert jobs == [] and m.seqs[d].base == [0, 1]
    assert m.seqs[d].res == [4, 5]               # fresh residual pages for the inherited prefix
    assert m.append(d, 5) == []                  # aligned: new page, nothing to copy
    e, jobs = m.fork(d, 37, share_res=True)      # copies d's 5-row tail, base and residual
    assert [(j[2], j[3]) for j in jobs] == [(5, JOB_BASE), (5, JOB_RES)]
    assert m.append(e, 3) == []                  # e owns its tail privately: nothing to copy


def test_append_copies_shared_partial_page():
    m = AllocatorModel(16, 16, P)
    a = m.seq_create(20)          # base [0, 1], res [0, 1]
    # share the partial page by hand through refcounts: fork at a full length never shares a
    # partial page under the pack policy, so emulate a frozen tail by bumping the refcount
    m.base_ref[1] += 1
    jobs = m.append(a, 1)
    assert jobs == [(1, 2, 4, JOB_BASE)]
    assert m.seqs[a].base == [0, 2] and m.base_ref[1] == 1


def test_errors_change_nothing():
    m = AllocatorModel(4, 4, P)
    a = m.seq_create(64)
    with pytest.raises(AllocatorError) as e:
        m.seq_create(1)
    assert e.value.code == ERR_OUT_OF_PAGES
    with pytest.raises(AllocatorError) as e:
        m.fork(a, 65)
    assert e.value.code == ERR_INVALID_ARG
    with pytest.raises(AllocatorError) as e:
        m.fork(a, 17)             # needs a tail page and 2 residual pages: none free
    assert e.value.code == ERR_OUT_OF_PAGES
    assert m.stats()["base_refsum"] == 4 and len(m.seqs) == 1
    with pytest.raises(AllocatorError) as e:
        m.free(99)
    assert e.value.code == ERR_INVALID_ARG


def test_commit_worked_example():
    """LCP commit (ForkServe README, "Methods"), worked by hand with the LIFO policy: two
    speculative branches of a 40-token root; branch b1 grows to 50 tokens; the observed tokens
    confirm only its first 20, inside the trunk's shared page 1, so that page is split."""
    m = AllocatorModel(16, 16, P)
    root = m.seq_create(40)                    # base [0, 1, 2], res [0, 1, 2]
    b1, _ = m.fork(root, 40)                   # base [0, 1, 3] (tail copy), res [3, 4, 5]
    b2, _ = m.fork(root, 40)                   # base [0, 1, 4], res [6, 7, 8]
    assert m.append(b1, 10) == []              # base [0, 1, 3, 5], res [3, 4, 5, 9]
    jobs = m.commit(b1, 20, siblings=[b2])
    # b2 frees base 4 and res 6, 7, 8; truncation frees base 3, 5 and res 5, 9; base page 1 is
    # still shared with the root, so b1 gets the last freed base page (5) with 20 % 16 = 4 rows
    assert jobs == [(1, 5, 4, JOB_BASE)]
    assert m.seqs[b1].base == [0, 5] and m.seqs[b1].res == [3, 4] and m.seqs[b1].length == 20
    assert b2 not in m.seqs
    assert m.base_free[-2:] == [4, 3] and m.res_free[-5:] == [6, 7, 8, 5, 9]
    assert m.base_ref[0] == 2 and m.base_ref[1] == 1 and m.base_ref[2] == 1
    # abort of the root now releases its own pages only: base 1 and 2 (page 0 is still b1's)
    # and its three residual pages
    assert m.abort(root) == (2, 3)
    assert m.base_ref[0] == 1


def test_commit_aborts_siblings_before_splitting():
    """A boundary page shared only with an aborted sibling is not copied."""
    m = AllocatorModel(16, 16, P)
    t = m.seq_create(32)                       # base [0, 1]
    a, _ = m.fork(t, 32)                       # aliases [0, 1]
    b, _ = m.fork(t, 32)
    m.free(t)                                  # trunk pages now shared by a and b only
    assert m.commit(a, 20, siblings=[b]) == []  # page 1 back to refcount 1: no split
    assert m.seqs[a].base == [0, 1] and m.base_ref[1] == 1
    c, _ = m.fork(a, 16)
    # truncation to 8 tokens releases page 1 (pushed on the free stack), then page 0, shared
    # with c, is split into the page on top of the stack: page 1 again
    assert m.commit(a, 8) == [(0, 1, 8, JOB_BASE)]
    assert m.seqs[a].base == [1] and m.seqs[c].base == [0] and m.base_ref[0] == 1


def test_commit_page_aligned_and_full_length():
    m = AllocatorModel(16, 16, P)
    r = m.seq_create(48)
    assert m.commit(r, 48) == [] and m.seqs[r].base == [0, 1, 2]
    assert m.commit(r, 32) == [] and m.seqs[r].base == [0, 1] and m.base_free[-1] == 2
    assert m.commit(r, 0) == [] and m.seqs[r].base == [] and m.seqs[r].length == 0
    assert m.append(r, 17) == [] and len(m.seqs[r].base) == 2


def test_abort_costs_the_residual_not_the_trunk():
    """ForkServe README, "Design vs APC": abort releases the branch's own pages; the trunk,
    aliased by the other branches, only loses a reference."""
    m = AllocatorModel(64, 64, P)
    root = m.seq_create(64)                    # 4 trunk pages
    kids = []
    for _ in range(4):
        c, _ = m.fork(root, 64)
        m.append(c, 20)                        # 2 own base pages, 4 + 2 own residual pages
        kids.append(c)
    live_before = m.stats()["base_live"]
    assert m.abort(kids[0]) == (2, 6)
    assert m.stats()["base_live"] == live_before - 2
    assert all(m.base_ref[p] == 4 for p in m.seqs[root].base)


def test_commit_errors_change_nothing():
    m = AllocatorModel(3, 12, P)
    a = m.seq_create(48)                       # base [0, 1, 2]: the base pool is empty
    c, _ = m.fork(a, 48)                       # aligned: aliases all three
    before = m._snapshot()

    def same():
        after = m._snapshot()
        return (after[0], after[1], after[2], after[3]) == (before[0], before[1], before[2], before[3]) and \
            {k: (v.length, v.base, v.res) for k, v in after[4].items()} == \
            {k: (v.length, v.base, v.res) for k, v in before[4].items()}

    for args, code in [((a, 49, []), ERR_INVALID_ARG), ((a, 20, [a]), ERR_INVALID_ARG),
                       ((a, 20, [c, c]), ERR_INVALID_ARG), ((a, 20, [99]), ERR_INVALID_ARG),
                       ((a, -1, []), ERR_INVALID_ARG)]:
        with pytest.raises(AllocatorError) as e:
            m.commit(*args)
        assert e.value.code == code and same()
    # truncating a to 20 tokens drops its reference to page 2 (c still holds it, nothing is
    # freed), and page 1, shared with c, needs a copy: no free base page
    with pytest.raises(AllocatorError) as e:
        m.commit(a, 20)
    assert e.value.code == ERR_OUT_OF_PAGES and same()
    # with c aborted first nothing is shared any more: no copy, page 2 freed
    assert m.commit(a, 20, siblings=[c]) == []
    assert m.base_free == [2] and m.seqs[a].base == [0, 1]


def test_lcp_len_pins():
    assert lcp_len([], [1, 2]) == 0
    assert lcp_len([5, 6, 7], [5, 6, 7]) == 3
    assert lcp_len([5, 6, 7, 8], [5, 6, 9]) == 2
    assert lcp_len([1], [2]) == 0
    assert lcp_len([3, 3, 3], [3, 3, 3, 3, 3]) == 3


def test_freeze_fork_worked_example():
    """Freeze-tail fork (ForkServe README, adaptive unaligned tail), worked by hand."""
    m = AllocatorModel(64, 64, P)
    root = m.seq_create(40)                    # base [0, 1, 2] (page 2 holds 8 rows), res [0, 1, 2]
    c1, jobs = m.fork(root, 40, freeze=True)   # aliases page 2 too; hole = slots 40..47
    # rows 8..15 of page 2 hold no token yet: zeroed; the child's own residual page 5 likewise
    assert jobs == [(2, 2, 8, JOB_BASE_ZERO), (5, 5, 8, JOB_RES_ZERO)]
    assert m.seqs[c1].base == [0, 1, 2] and m.seqs[c1].res == [3, 4, 5]
    assert m.slot_maps([c1]) == [(40, 8)] and m.page_tables([c1], 3)[2] == [48]
    c2, jobs = m.fork(root, 40, freeze=True)
    assert jobs == [(2, 2, 8, JOB_BASE_ZERO), (8, 8, 8, JOB_RES_ZERO)]
    assert m.base_ref[2] == 3 and m.stats()["base_live"] == 3  # no tail copies
    assert m.append(c1, 5) == [] and m.seqs[c1].base == [0, 1, 2, 3]  # own tokens start on a new page
    # the parent keeps writing its frozen tail in place (the children read only rows 0..7)
    assert m.append(root, 4) == [] and m.seqs[root].base == [0, 1, 2]
    c3, jobs = m.fork(root, 44, freeze=True)   # rows 12..15 are still empty
    assert jobs[0] == (2, 2, 12, JOB_BASE_ZERO) and m.slot_maps([c3]) == [(44, 4)]
    assert m.append(root, 1) == [] and m.seqs[root].base == [0, 1, 2]
    # a child that commits back into the shared page no longer has a hole and gets its own copy
    assert m.commit(c2, 36) == [(2, 4, 4, JOB_BASE)]
    assert m.slot_maps([c2]) == [(0, 0)] and m.page_tables([c2], 3)[2] == [36]
    # a freeze fork of a child whose prefix spans its hole is a pack fork that inherits the hole
    g, jobs = m.fork(c1, 42, freeze=True)
    assert m.slot_maps([g]) == [(40, 8)] and jobs == [(3, jobs[0][1], 2, JOB_BASE)]
    # freeing the parent hands the frozen page to nobody: a later append by a child copies nothing
    m.free(root)                               # page 2 stays with c1, c3 and g
    assert m.base_ref[2] == 3 and m.owner[JOB_BASE][2] == -1


@pytest.mark.parametrize("L,k,ell", [(2050, 4, 48), (2047, 8, 100), (40, 3, 16), (4096, 4, 7)])
def test_freeze_page_count_matches_formula(L, k, ell):
    """pages_freeze = 1 + k ceil(l / P) pages beyond the trunk's full pages (ForkServe README)."""
    m = AllocatorModel(100000, 100000, P)
    root = m.seq_create(L)
    for _ in range(k):
        c, _ = m.fork(root, L, freeze=True)
        m.append(c, ell)
    full = L // P
    if L % P:
        assert m.stats()["base_live"] == full + acc.pages_freeze_children(L, k, ell, P)
    else:
        assert m.stats()["base_live"] == full + k * math.ceil(ell / P)
