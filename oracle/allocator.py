"""Pure-Python model of the paged, refcounted fork allocator (test infrastructure only).

Restates, as plain list manipulation:
* ForkKV L2, section 3 (Figure 6, fork analogy): a new agent maps its parent's
  base-cache pages read-only and pays only for its own residual pages;
* ForkServe README, "Design vs APC" and "Methods" (CoW tree): fork aliases the
  parent's page frames at once; live memory is b(L + sum l_i), not b(kL + sum l_i);
  freeing the parent does not drop the trunk (the child's reference pins it);
* ForkServe README, adaptive unaligned tail and "Status": the pack path clones
  the r = L mod P valid rows of the parent's partial last page into a private
  page of the child (a row copy of n_valid rows, not P);
* ForkServe README, "Methods" (LCP commit; CoW tree: abort costs the residual,
  not the trunk): a committed branch keeps the observed token prefix, its
  siblings are aborted, and a boundary page in the middle of a shared page is
  split copy-on-write;
* ForkServe README, adaptive unaligned tail (pages_freeze = 1 + k ceil(l/P):
  one read-only tail page shared by the k children; "freeze-tail needs a
  fork-aware slot map"): with the freeze flag a child aliases the parent's
  partial tail page too, and its own tokens start on a fresh page, leaving a
  hole in its slots.

Policies the pages leave open (fixed here so page ids are deterministic, and
mirrored bit for bit by the C++ allocator):
* each pool has a LIFO free stack, initialised so that pops yield 0, 1, 2, ...;
* freeing walks base pages then residual pages in logical order, pushing a page
  when its refcount reaches zero;
* fork without FORK_SHARE_RES allocates fresh residual pages for the whole
  inherited prefix (the child's adapter gives it different xA rows); with it,
  full residual pages are aliased and a partial one is copied like the base tail;
* append copies a partial last page first if it is shared (refcount > 1);
* commit aborts the siblings first (each like free, in the order given), then
  drops the branch's pages past the committed prefix (base then residual, in
  logical order), then splits the boundary page of each pool only if it is
  still shared, base before residual;
* sequence ids count up from 0 and are never reused;
* on any error nothing changes;
* slots: token p of a sequence sits in slot p, or p + hole length if the
  sequence has a hole and p is at or past its first slot; pages cover slots;
  page tables report slot counts;
* a freeze fork applies only to an unaligned prefix that does not span the
  parent's hole (else it is a pack fork, and the child inherits that hole); the
  shared tail page remembers the most rows any child reads ("frozen rows") and
  its owner (the parent, while that page is its partial tail and it holds it),
  which alone appends into it in place, past the frozen rows; zero jobs clear
  the page's rows no token has reached yet and the hole rows of the child's own
  residual page (or of the shared residual tail page with FORK_SHARE_RES).
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

OK = 0
ERR_INVALID_ARG = -1
ERR_OUT_OF_PAGES = -2
ERR_BAD_PAGE = -3
ERR_REFCOUNT = -4
ERR_UNSUPPORTED = -5

JOB_BASE = 0
JOB_RES = 1
JOB_BASE_ZERO = 2
JOB_RES_ZERO = 3


class AllocatorError(Exception):
    def __init__(self, code: int, msg: str = ""):
        super().__init__(f"{code}: {msg}")
        self.code = code


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class _Seq:
    __slots__ = ("length", "base", "res", "hole_start", "hole_len")

    def __init__(self, length: int, base: List[int], res: List[int], hole_start: int = 0, hole_len: int = 0):
        self.length = length
        self.base = base
        self.res = res
        self.hole_start = hole_start
        self.hole_len = hole_len

    def slots(self) -> int:
        return self.length + self.hole_len

    def slots_of(self, n: int) -> int:
        """Slots taken by the first n tokens."""
        return n + self.hole_len if self.hole_len and n > self.hole_start else n


class AllocatorModel:
    def __init__(self, num_base_pages: int, num_res_pages: int, page_size: int):
        if num_base_pages < 0 or num_res_pages < 0 or page_size < 1:
            raise AllocatorError(ERR_INVALID_ARG, "bad pool sizes")
        self.P = page_size
        self.base_free = list(range(num_base_pages - 1, -1, -1))
        self.res_free = list(range(num_res_pages - 1, -1, -1))
        self.base_ref = [0] * num_base_pages
        self.res_ref = [0] * num_res_pages
        self.frozen = {JOB_BASE: [0] * num_base_pages, JOB_RES: [0] * num_res_pages}
        self.owner = {JOB_BASE: [-1] * num_base_pages, JOB_RES: [-1] * num_res_pages}
        self.seqs: Dict[int, _Seq] = {}
        self.next_id = 0

    # -- helpers -----------------------------------------------------------
    def _seq(self, sid: int) -> _Seq:
        if sid not in self.seqs:
            raise AllocatorError(ERR_INVALID_ARG, f"unknown sequence {sid}")
        return self.seqs[sid]

    def _pop(self, kind: int) -> int:
        stack, ref = (self.base_free, self.base_ref) if kind == JOB_BASE else (self.res_free, self.res_ref)
        p = stack.pop()
        ref[p] = 1
        self.frozen[kind][p] = 0
        self.owner[kind][p] = -1
        return p

    def _release(self, kind: int, p: int, sid: int) -> None:
        """sid drops its reference to page p."""
        stack, ref = (self.base_free, self.base_ref) if kind == JOB_BASE else (self.res_free, self.res_ref)
        if self.owner[kind][p] == sid:
            self.owner[kind][p] = -1
        ref[p] -= 1
        if ref[p] == 0:
            stack.append(p)
            self.frozen[kind][p] = 0
            self.owner[kind][p] = -1

    def _in_place(self, kind: int, p: int, sid: int, row: int) -> bool:
        """sid may write rows >= row of its shared page p: its own frozen tail, past the frozen rows."""
        return self.owner[kind][p] == sid and row >= self.frozen[kind][p]

    def _new_id(self) -> int:
        sid = self.next_id
        self.next_id += 1
        return sid

    # -- operations --------------------------------------------------------
    def seq_create(self, n_tokens: int) -> int:
        if n_tokens < 0:
            raise AllocatorError(ERR_INVALID_ARG, "negative length")
        npg = _ceil_div(n_tokens, self.P)
        if npg > len(self.base_free) or npg > len(self.res_free):
            raise AllocatorError(ERR_OUT_OF_PAGES)
        base = [self._pop(JOB_BASE) for _ in range(npg)]
        res = [self._pop(JOB_RES) for _ in range(npg)]
        sid = self._new_id()
        self.seqs[sid] = _Seq(n_tokens, base, res)
        return sid

    def fork(self, parent: int, prefix_len: int, share_res: bool = False, freeze: bool = False,
             jobs_cap: Optional[int] = None) -> Tuple[int, List[Tuple[int, int, int, int]]]:
        par = self._seq(parent)
        if prefix_len < 0 or prefix_len > par.length:
            raise AllocatorError(ERR_INVALID_ARG, "prefix_len out of range")
        P = self.P
        inherit = bool(par.hole_len) and prefix_len > par.hole_start
        slot_end = par.slots_of(prefix_len)
        nf, t = divmod(slot_end, P)
        npg = nf + (1 if t else 0)
        frz = freeze and t != 0 and not inherit
        written = min(par.slots() - nf * P, P) if frz else P   # rows of the tail page with tokens
        if frz:
            need_base = 0
            need_res = 0 if share_res else npg
            n_jobs = (1 if written < P else 0) + ((1 if written < P else 0) if share_res else 1)
        else:
            need_base = 1 if t else 0
            need_res = (1 if t else 0) if share_res else npg
            n_jobs = (1 if t else 0) * (2 if share_res else 1)
        if jobs_cap is not None and n_jobs > jobs_cap:
            raise AllocatorError(ERR_INVALID_ARG, "job buffer too small")
        if need_base > len(self.base_free) or need_res > len(self.res_free):
            raise AllocatorError(ERR_OUT_OF_PAGES)
        jobs = []
        hole = (par.hole_start, par.hole_len) if inherit else (0, 0)
        base = list(par.base[:nf])
        for p in base:
            self.base_ref[p] += 1
        if frz:
            tp = par.base[nf]
            base.append(tp)
            self.base_ref[tp] += 1
            self.frozen[JOB_BASE][tp] = max(self.frozen[JOB_BASE][tp], t)
            if self.owner[JOB_BASE][tp] < 0 and par.slots() < (nf + 1) * P:
                self.owner[JOB_BASE][tp] = parent
            if written < P:
                jobs.append((tp, tp, written, JOB_BASE_ZERO))
            hole = (slot_end, P - t)
            if share_res:
                res = list(par.res[:nf + 1])
                for p in res:
                    self.res_ref[p] += 1
                rp = par.res[nf]
                self.frozen[JOB_RES][rp] = max(self.frozen[JOB_RES][rp], t)
                if self.owner[JOB_RES][rp] < 0 and par.slots() < (nf + 1) * P:
                    self.owner[JOB_RES][rp] = parent
                if written < P:
                    jobs.append((rp, rp, written, JOB_RES_ZERO))
            else:
                res = [self._pop(JOB_RES) for _ in range(npg)]
                jobs.append((res[nf], res[nf], t, JOB_RES_ZERO))
        else:
            if t:
                dst = self._pop(JOB_BASE)
                jobs.append((par.base[nf], dst, t, JOB_BASE))
                base.append(dst)
            if share_res:
                res = list(par.res[:nf])
                for p in res:
                    self.res_ref[p] += 1
                if t:
                    dst = self._pop(JOB_RES)
                    jobs.append((par.res[nf], dst, t, JOB_RES))
                    res.append(dst)
            else:
                res = [self._pop(JOB_RES) for _ in range(npg)]
        sid = self._new_id()
        self.seqs[sid] = _Seq(prefix_len, base, res, hole[0], hole[1])
        return sid, jobs

    def append(self, sid: int, n_tokens: int, jobs_cap: Optional[int] = None) -> List[Tuple[int, int, int, int]]:
        s = self._seq(sid)
        if n_tokens < 0:
            raise AllocatorError(ERR_INVALID_ARG, "negative length")
        P = self.P
        S = s.slots()
        grow = _ceil_div(S + n_tokens, P) - _ceil_div(S, P)
        tail = S % P
        cow_base = bool(n_tokens > 0 and tail and self.base_ref[s.base[-1]] > 1
                        and not self._in_place(JOB_BASE, s.base[-1], sid, tail))
        cow_res = bool(n_tokens > 0 and tail and self.res_ref[s.res[-1]] > 1
                       and not self._in_place(JOB_RES, s.res[-1], sid, tail))
        n_jobs = int(cow_base) + int(cow_res)
        if jobs_cap is not None and n_jobs > jobs_cap:
            raise AllocatorError(ERR_INVALID_ARG, "job buffer too small")
        if grow + cow_base > len(self.base_free) or grow + cow_res > len(self.res_free):
            raise AllocatorError(ERR_OUT_OF_PAGES)
        jobs = []
        if cow_base:
            old = s.base[-1]
            dst = self._pop(JOB_BASE)
            self._release(JOB_BASE, old, sid)
            s.base[-1] = dst
            jobs.append((old, dst, tail, JOB_BASE))
        s.base.extend(self._pop(JOB_BASE) for _ in range(grow))
        if cow_res:
            old = s.res[-1]
            dst = self._pop(JOB_RES)
            self._release(JOB_RES, old, sid)
            s.res[-1] = dst
            jobs.append((old, dst, tail, JOB_RES))
        s.res.extend(self._pop(JOB_RES) for _ in range(grow))
        s.length += n_tokens
        return jobs

    def free(self, sid: int) -> None:
        s = self._seq(sid)
        for p in s.base:
            self._release(JOB_BASE, p, sid)
        for p in s.res:
            self._release(JOB_RES, p, sid)
        del self.seqs[sid]

    def abort(self, sid: int) -> Tuple[int, int]:
        """Free a speculative branch; return how many base and residual pages went back to the pool."""
        s = self._seq(sid)
        nb = sum(1 for p in s.base if self.base_ref[p] == 1)
        nr = sum(1 for p in s.res if self.res_ref[p] == 1)
        self.free(sid)
        return nb, nr

    def _snapshot(self):
        return (list(self.base_free), list(self.res_free), list(self.base_ref), list(self.res_ref),
                {k: _Seq(v.length, list(v.base), list(v.res), v.hole_start, v.hole_len) for k, v in self.seqs.items()},
                {k: list(v) for k, v in self.frozen.items()}, {k: list(v) for k, v in self.owner.items()})

    def _restore(self, snap) -> None:
        (self.base_free, self.res_free, self.base_ref, self.res_ref, self.seqs, self.frozen, self.owner) = snap

    def commit(self, sid: int, lcp_len: int, siblings: Sequence[int] = (),
               jobs_cap: Optional[int] = None) -> List[Tuple[int, int, int, int]]:
        """LCP commit: abort the siblings, keep the first lcp_len tokens of sid, split a shared boundary page."""
        s = self._seq(sid)
        if lcp_len < 0 or lcp_len > s.length:
            raise AllocatorError(ERR_INVALID_ARG, "lcp_len out of range")
        sibs = list(siblings)
        if sid in sibs or len(set(sibs)) != len(sibs):
            raise AllocatorError(ERR_INVALID_ARG, "bad sibling list")
        for o in sibs:
            self._seq(o)
        snap = self._snapshot()
        try:
            for o in sibs:
                self.free(o)
            s = self.seqs[sid]
            P = self.P
            n_slots = s.slots_of(lcp_len)   # the hole goes as well if the prefix ends at or before it
            keep = _ceil_div(n_slots, P)
            t = n_slots % P
            for p in s.base[keep:]:
                self._release(JOB_BASE, p, sid)
            for p in s.res[keep:]:
                self._release(JOB_RES, p, sid)
            del s.base[keep:]
            del s.res[keep:]
            split_b = bool(t) and self.base_ref[s.base[-1]] > 1 and not self._in_place(JOB_BASE, s.base[-1], sid, t)
            split_r = bool(t) and self.res_ref[s.res[-1]] > 1 and not self._in_place(JOB_RES, s.res[-1], sid, t)
            if jobs_cap is not None and int(split_b) + int(split_r) > jobs_cap:
                raise AllocatorError(ERR_INVALID_ARG, "job buffer too small")
            if (split_b and not self.base_free) or (split_r and not self.res_free):
                raise AllocatorError(ERR_OUT_OF_PAGES)
            jobs = []
            if split_b:
                old = s.base[-1]
                dst = self._pop(JOB_BASE)
                self._release(JOB_BASE, old, sid)
                s.base[-1] = dst
                jobs.append((old, dst, t, JOB_BASE))
            if split_r:
                old = s.res[-1]
                dst = self._pop(JOB_RES)
                self._release(JOB_RES, old, sid)
                s.res[-1] = dst
                jobs.append((old, dst, t, JOB_RES))
            if s.hole_len and lcp_len <= s.hole_start:
                s.hole_start = s.hole_len = 0
            s.length = lcp_len
            return jobs
        except AllocatorError:
            self._restore(snap)
            raise

    def page_tables(self, sids: Sequence[int], stride: int):
        """Rows of base / residual page ids (padded with -1) and lengths in slots."""
        bpt, rpt, lens = [], [], []
        for sid in sids:
            s = self._seq(sid)
            if len(s.base) > stride:
                raise AllocatorError(ERR_INVALID_ARG, "stride too small")
            bpt.append(s.base + [-1] * (stride - len(s.base)))
            rpt.append(s.res + [-1] * (stride - len(s.res)))
            lens.append(s.slots())
        return bpt, rpt, lens

    def slot_maps(self, sids: Sequence[int]) -> List[Tuple[int, int]]:
        return [(self._seq(sid).hole_start, self._seq(sid).hole_len) for sid in sids]

    def refcount(self, kind: int, page: int) -> int:
        ref = self.base_ref if kind == JOB_BASE else self.res_ref
        if page < 0 or page >= len(ref):
            raise AllocatorError(ERR_BAD_PAGE)
        return ref[page]

    def stats(self) -> dict:
        return {
            "n_seqs": len(self.seqs),
            "base_live": sum(1 for c in self.base_ref if c > 0),
            "res_live": sum(1 for c in self.res_ref if c > 0),
            "base_free": len(self.base_free),
            "res_free": len(self.res_free),
            "base_shared": sum(1 for c in self.base_ref if c > 1),
            "res_shared": sum(1 for c in self.res_ref if c > 1),
            "base_refsum": sum(self.base_ref),
            "res_refsum": sum(self.res_ref),
        }


def lcp_len(spec: Sequence[int], observed: Sequence[int]) -> int:
    """Tokens of a speculative branch confirmed by the observed sequence (longest common prefix)."""
    n = 0
    while n < len(spec) and n < len(observed) and spec[n] == observed[n]:
        n += 1
    return n


def cow_copy_rows_model(src_page_rows, dst_page_rows, n_valid: int):
    """Row copy of the pack path: rows [0, n_valid) of src into dst, the rest untouched."""
    out = [list(r) for r in dst_page_rows]
    for i in range(n_valid):
        out[i] = list(src_page_rows[i])
    return out
