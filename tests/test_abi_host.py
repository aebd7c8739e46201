"""Host-side checks of libforkkv (no GPU needed).

* the shared library loads and exports every function include/forkkv.h declares;
* the C++ allocator matches the pure-Python allocator model bit for bit (page
  ids, jobs, refcounts, stats) on the ForkServe scenarios and on random
  operation sequences, including the no-change-on-error rule;
* the decode work plan covers every (agent, logical page) exactly once, only
  groups agents that map the same physical page, and lists each agent's slots.
"""
import os
import random
import re

import numpy as np
import pytest

from disaggregated_kv_attention_gb300 import forkkv as fk
from oracle.allocator import AllocatorError, AllocatorModel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    from disaggregated_kv_attention_gb300 import build
    build.build()
    return fk.lib()


def test_exports_every_declared_function():
    with open(os.path.join(ROOT, "include", "forkkv.h")) as f:
        text = f.read()
    names = set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(forkkv_\w+)\s*\(", text, flags=re.M))
    assert len(names) >= 20, names
    lib = fk.lib()
    missing = [n for n in sorted(names) if not hasattr(lib, n)]
    assert not missing, missing
    assert set(fk._SIGNATURES) == names  # the binding declares exactly the header's functions


def test_strerror_and_version():
    assert fk.strerror(0) == "ok"
    assert "pages" in fk.strerror(-2)
    assert fk.lib().forkkv_version() >= 100


class _Pair:
    """C++ allocator and Python model driven side by side."""

    def __init__(self, nb, nr):
        self.c = fk.forkkv_alloc_create(nb, nr)
        self.m = AllocatorModel(nb, nr, 16)
        self.ids = {}  # model id -> C id (they must be equal)

    def close(self):
        fk.forkkv_alloc_destroy(self.c)

    def op(self, name, *args):
        err_c = err_m = None
        rc = rm = None
        try:
            rc = getattr(self, "_c_" + name)(*args)
        except fk.ForkKVError as e:
            err_c = e.code
        try:
            rm = getattr(self, "_m_" + name)(*args)
        except AllocatorError as e:
            err_m = e.code
        assert err_c == err_m, (name, args, err_c, err_m)
        assert rc == rm, (name, args, rc, rm)
        return rm

    def _c_create(self, n):
        return fk.forkkv_seq_create(self.c, n)

    def _m_create(self, n):
        return self.m.seq_create(n)

    def _c_fork(self, p, n, share, freeze=False):
        return fk.forkkv_fork(self.c, p, n, (fk.FORK_SHARE_RES if share else 0) | (fk.FORK_FREEZE_TAIL if freeze else 0))

    def _m_fork(self, p, n, share, freeze=False):
        return self.m.fork(p, n, share_res=share, freeze=freeze)

    def _c_append(self, s, n):
        return fk.forkkv_append(self.c, s, n)

    def _m_append(self, s, n):
        return self.m.append(s, n)

    def _c_free(self, s):
        return fk.forkkv_free(self.c, s)

    def _m_free(self, s):
        return self.m.free(s)

    def _c_commit(self, s, n, sibs):
        return fk.forkkv_commit(self.c, s, n, sibs)

    def _m_commit(self, s, n, sibs):
        return self.m.commit(s, n, sibs, jobs_cap=2)

    def _c_abort(self, s):
        return fk.forkkv_abort(self.c, s)

    def _m_abort(self, s):
        return self.m.abort(s)

    def check_state(self):
        st = fk.forkkv_stats_get(self.c)
        ms = self.m.stats()
        for k in ms:
            assert st[k] == ms[k], (k, st[k], ms[k])
        sids = sorted(self.m.seqs)
        if sids:
            stride = max(1, max(len(self.m.seqs[s].base) for s in sids))
            b, r, l = fk.forkkv_page_tables(self.c, sids, stride)
            mb, mr, ml = self.m.page_tables(sids, stride)
            assert np.array_equal(b, np.array(mb, np.int32))
            assert np.array_equal(r, np.array(mr, np.int32))
            assert np.array_equal(l, np.array(ml, np.int32))
            assert np.array_equal(fk.forkkv_slot_maps(self.c, sids), np.array(self.m.slot_maps(sids), np.int32))
        for p in range(0, len(self.m.base_ref), 7):
            assert fk.forkkv_refcount(self.c, fk.JOB_BASE, p) == self.m.base_ref[p]


def test_cpp_allocator_matches_model_on_forkserve_scenarios():
    for L, k, ell in [(2048, 4, 64), (4096, 8, 128), (2050, 4, 48), (8192, 8, 32), (1024, 6, 4), (16384, 4, 256)]:
        pr = _Pair(20000, 40000)
        root = pr.op("create", L)
        kids = []
        for _ in range(k):
            c, jobs = pr.op("fork", root, L, False)
            kids.append(c)
            pr.op("append", c, ell)
        pr.check_state()
        pr.op("free", root)
        pr.check_state()
        pr.close()


def test_cpp_allocator_matches_model_on_random_operations():
    rnd = random.Random(11)
    pr = _Pair(200, 260)
    live = []
    for step in range(2500):
        x = rnd.random()
        if x < 0.2 or not live:
            sid = pr.op("create", rnd.randint(0, 60))
            if sid is not None:
                live.append(sid)
        elif x < 0.5:
            par = rnd.choice(live)
            res = pr.op("fork", par, rnd.randint(0, pr.m.seqs[par].length + 2), rnd.random() < 0.3,
                        rnd.random() < 0.4)
            if res is not None:
                live.append(res[0])
        elif x < 0.8:
            pr.op("append", rnd.choice(live), rnd.randint(-1, 40))
        else:
            pr.op("free", live.pop(rnd.randrange(len(live))))
        if step % 50 == 0:
            pr.check_state()
    pr.check_state()
    for s in live:
        pr.op("free", s)
    st = fk.forkkv_stats_get(pr.c)
    assert st["base_free"] == 200 and st["res_free"] == 260 and st["n_seqs"] == 0
    pr.close()


def test_cpp_commit_and_abort_match_model():
    """Speculative fan-outs committed at random common prefixes (some inside shared pages,
    some with bad arguments) and aborted branches: same ids, jobs, tables and free stacks."""
    rnd = random.Random(23)
    pr = _Pair(160, 400)
    live = []
    seen = {"split": 0, "rejected": 0}
    for step in range(3000):
        x = rnd.random()
        if x < 0.12 or not live:
            sid = pr.op("create", rnd.randint(0, 70))
            if sid is not None:
                live.append(sid)
        elif x < 0.42:
            par = rnd.choice(live)
            res = pr.op("fork", par, rnd.randint(0, pr.m.seqs[par].length), rnd.random() < 0.3, rnd.random() < 0.4)
            if res is not None:
                live.append(res[0])
        elif x < 0.62:
            pr.op("append", rnd.choice(live), rnd.randint(0, 30))
        elif x < 0.84:
            s = rnd.choice(live)
            others = [o for o in live if o != s]
            sibs = rnd.sample(others, min(len(others), rnd.randint(0, 3)))
            if rnd.random() < 0.05 and sibs:
                sibs.append(sibs[0])                  # a repeated sibling: rejected
            if rnd.random() < 0.05:
                sibs.append(s)                        # the branch itself: rejected
            n = rnd.randint(-1, pr.m.seqs[s].length + 1)
            jobs = pr.op("commit", s, n, sibs)
            if jobs is None:
                seen["rejected"] += 1
            else:
                seen["split"] += bool(jobs)
                live = [o for o in live if o not in sibs]
        else:
            pr.op("abort", live.pop(rnd.randrange(len(live))))
        if step % 40 == 0:
            pr.check_state()
    pr.check_state()
    assert seen["split"] > 20 and seen["rejected"] > 20, seen
    for s in live:
        pr.op("abort", s)
    st = fk.forkkv_stats_get(pr.c)
    assert st["base_free"] == 160 and st["res_free"] == 400 and st["n_seqs"] == 0
    pr.close()


def test_lcp_len_matches_model():
    from oracle.allocator import lcp_len
    rnd = random.Random(3)
    for _ in range(300):
        n = rnd.randint(0, 12)
        a = [rnd.randint(0, 3) for _ in range(n)]
        b = a[:rnd.randint(0, n)] + [rnd.randint(0, 3) for _ in range(rnd.randint(0, 5))]
        assert fk.forkkv_lcp_len(a, b) == lcp_len(a, b)


def test_invalid_arguments_rejected():
    a = fk.forkkv_alloc_create(8, 8)
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_free(a, 123)
    assert e.value.code == -1
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_refcount(a, fk.JOB_BASE, 8)
    assert e.value.code == -3
    with pytest.raises(fk.ForkKVError) as e:
        fk.forkkv_alloc_create(8, 8, 32)
    assert e.value.code == -5
    fk.forkkv_alloc_destroy(a)
    for polls in (0, (1 << 20) + 1):  # rejected before any CUDA call: nothing is launched
        with pytest.raises(fk.ForkKVError) as e:
            fk.forkkv_wait_selftest(polls, stream=0)
        assert e.value.code == -1


def _tree_tables(rnd, n_agents_per, depth_tokens):
    """Page tables of a random two-level fork tree built with the C++ allocator."""
    a = fk.forkkv_alloc_create(100000, 200000)
    root = fk.forkkv_seq_create(a, depth_tokens[0])
    agents = []
    for t in range(len(n_agents_per)):
        trunk, _ = fk.forkkv_fork(a, root, depth_tokens[0])
        fk.forkkv_append(a, trunk, depth_tokens[1])
        L = depth_tokens[0] + depth_tokens[1]
        for _ in range(n_agents_per[t]):
            c, _ = fk.forkkv_fork(a, trunk, L)
            fk.forkkv_append(a, c, rnd.randint(1, 300))
            agents.append(c)
    stride = max(fk.forkkv_seq_len(a, s) for s in agents) // 16 + 1
    bpt, rpt, lens = fk.forkkv_page_tables(a, agents, stride)
    fk.forkkv_alloc_destroy(a)
    return bpt, lens


@pytest.mark.parametrize("shape", [([3], (512, 0)), ([16, 16, 16, 16], (4096, 256)), ([1, 9, 5], (200, 37)),
                                   ([2], (0, 0))])
@pytest.mark.parametrize("target", [0, 7, 1000])
def test_plan_covers_every_page_once(shape, target):
    rnd = random.Random(5)
    per, toks = shape
    bpt, lens = _tree_tables(rnd, per, toks)
    A = len(lens)
    hkv = 8
    plan, info = fk.forkkv_plan_build(bpt, lens, hkv, target)
    items = plan[:info.n_items * fk.PLAN_ITEM_INTS].reshape(info.n_items, fk.PLAN_ITEM_INTS)
    off = plan[info.n_items * fk.PLAN_ITEM_INTS:][:A + 1]
    rest = plan[info.n_items * fk.PLAN_ITEM_INTS + A + 1:]
    slots, units = rest[:info.n_slots], rest[info.n_slots:]
    assert info.plan_ints == plan.size and units.size == info.n_units * fk.PLAN_UNIT_INTS
    assert info.n_units == info.n_items * hkv
    units = units.reshape(info.n_units, fk.PLAN_UNIT_INTS)
    # the schedule: at most target (152 for 0) CTAs, none idle, every (item, head) unit once,
    # each record a copy of its item's fields
    assert 1 <= info.n_ctas <= (target or 152)
    by_slot = {it[12]: i for i, it in enumerate(items)}
    records, pairs, loads = set(), set(), []
    cost = lambda it: ((it[1] - it[0] + 7) // 8) * max(930 * it[2], 2400) + 3000
    for c in range(info.n_ctas):
        r, load = c, 0
        while r != -1:
            assert 0 <= r < info.n_units and r not in records and (r < info.n_ctas) == (r == c)
            records.add(r)
            u = units[r]
            i = by_slot[u[4]]
            it = items[i]
            assert list(u[:3]) == list(it[:3]) and list(u[6:10]) == list(it[4:8]) and not u[10:].any()
            assert 0 <= u[3] < hkv and (i, u[3]) not in pairs
            pairs.add((i, u[3]))
            load += cost(it)
            r = u[5]
        loads.append(load)
    assert len(records) == len(pairs) == info.n_units
    # greedy list scheduling bound: no CTA ends later than the mean load plus one unit
    all_costs = [cost(it) for it in items] * hkv
    assert max(loads) <= sum(all_costs) / info.n_ctas + max(all_costs)
    cover = {}
    slot_owner = {}
    for i, it in enumerate(items):
        p0, p1, na, wpp = it[:4]
        assert na in (1, 2, 4) and wpp == 8 and 0 <= p0 < p1
        ags = list(it[4:4 + na])
        for x, ag in enumerate(ags):
            slot_owner[it[12] + x] = ag
        for pg in range(p0, p1):
            phys = {bpt[ag, pg] for ag in ags}
            assert len(phys) == 1  # one base page read for all agents of the item
            for ag in ags:
                assert pg < (lens[ag] + 15) // 16
                assert (ag, pg) not in cover
                cover[(ag, pg)] = i
    for ag in range(A):
        for pg in range((lens[ag] + 15) // 16):
            assert (ag, pg) in cover
        assert sorted(slots[off[ag]:off[ag + 1]]) == sorted(s for s, o in slot_owner.items() if o == ag)
    assert off[A] == info.n_slots



def test_cpp_freeze_fanout_matches_model():
    """Same-batch fan-outs of unaligned trunks with the freeze flag, the parent writing on, children
    appending, committing and aborting: ids, jobs (copies and zero jobs), tables, slot maps."""
    for L, k, ell in [(2050, 4, 48), (40, 6, 3), (16, 3, 20), (1000, 8, 200)]:
        pr = _Pair(4000, 8000)
        root = pr.op("create", L)
        kids = []
        for i in range(k):
            c, jobs = pr.op("fork", root, L, i % 2 == 1, True)
            kids.append(c)
            pr.op("append", c, ell)
            pr.op("append", root, 1)
        pr.check_state()
        pr.op("commit", kids[0], L - 1, kids[1:3])
        if k > 3:
            pr.op("abort", kids[3])
        pr.check_state()
        pr.op("free", root)
        pr.check_state()
        pr.close()


def test_plan_deals_sibling_groups_side_by_side():
    """Agent groups that read the same trunk pages (one segment, split into groups of 4) are dealt,
    for the same pages and KV head, to consecutive CTAs of the first round, so that they stream
    those pages at the same time (the planner's order: cost, segment, first block, head, group;
    each unit to the least loaded CTA, so CTA c's first unit is the c-th)."""
    rnd = random.Random(11)
    bpt, lens = _tree_tables(rnd, [16, 16], (4096, 256))  # 32 agents on one root, 2 trunks of 16
    hkv = 8
    plan, info = fk.forkkv_plan_build(bpt, lens, hkv, 0)
    items = plan[:info.n_items * fk.PLAN_ITEM_INTS].reshape(info.n_items, fk.PLAN_ITEM_INTS)
    rest = plan[info.n_items * fk.PLAN_ITEM_INTS + len(lens) + 1:]
    units = rest[info.n_slots:].reshape(info.n_units, fk.PLAN_UNIT_INTS)
    by_slot = {it[12]: i for i, it in enumerate(items)}
    cost = lambda it: ((it[1] - it[0] + 7) // 8) * max(930 * it[2], 2400) + 3000
    siblings = {}
    for c in range(info.n_ctas):  # record c is CTA c's first unit
        u = units[c]
        it = items[by_slot[u[4]]]
        p0, p1 = int(it[0]), int(it[1])
        key = (cost(it), p0, p1, int(bpt[it[4], p0]), int(u[3]))  # same pages (physical), same head
        siblings.setdefault(key, []).append((c, tuple(int(a) for a in it[4:4 + it[2]])))
    groups = [v for v in siblings.values() if len(v) > 1]
    assert groups, "the scenario must put sibling groups in the first round"
    for v in groups:
        cs = [c for c, _ in v]
        assert cs == list(range(cs[0], cs[0] + len(cs))), v  # consecutive CTAs
        agent_sets = [set(ags) for _, ags in v]
        assert all(not (x & y) for i, x in enumerate(agent_sets) for y in agent_sets[i + 1:])  # distinct groups
