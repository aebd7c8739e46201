// Host allocator: paged, refcounted base and residual pools with fork / append /
// free and copy-on-write jobs.
//
// Semantics: ForkKV L2 section 3 (Figure 6: a new agent maps the parent's base
// pages read-only and allocates only its residual pages) and the ForkServe
// README ("Design vs APC" and "Methods": fork aliases the parent's frames in
// O(pages) with refcounts, so freeing the parent keeps the trunk alive;
// unaligned tail: the pack path copies the L mod P valid rows into a private
// page of each child, the freeze path keeps one read-only tail page shared by
// the children, whose own tokens start on a fresh page (pages_freeze =
// 1 + k ceil(l / P)), which needs a fork-aware slot map: each child's slots
// skip the rest of the frozen page; "Methods", LCP commit: the committed branch
// keeps the observed prefix, a mid-page boundary is split copy-on-write and the
// siblings are aborted, which releases their own pages and only decrements the
// trunk's).  Free-list order, id assignment and the error policy are fixed
// choices documented in include/forkkv.h.
//
// Slots: a sequence's keys live in slots 0, 1, ... (slot s is row s % 16 of
// its page s / 16).  Token p sits in slot p, except in a sequence with a hole
// [hole_start, hole_start + hole_len) (made by a freeze fork), where tokens at
// or past hole_start sit hole_len slots further on.  Pages cover the slots.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/forkkv.h"

namespace {

struct Seq {
  int32_t length = 0;      // tokens
  int32_t hole_start = 0;  // first slot of the hole (0 with no hole)
  int32_t hole_len = 0;    // slots in the hole (0: none)
  std::vector<int32_t> base;
  std::vector<int32_t> res;
  int32_t slots() const { return length + hole_len; }
  // slots taken by the first n tokens
  int32_t slots_of(int32_t n) const { return hole_len && n > hole_start ? n + hole_len : n; }
};

inline int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

}  // namespace

struct forkkv_alloc {
  int32_t page = FORKKV_PAGE_SIZE;
  std::vector<int32_t> base_free, res_free;  // LIFO stacks
  std::vector<int32_t> base_ref, res_ref;
  // a page frozen by freeze forks: its rows [0, frozen) are read by the children; only its
  // owner (the sequence it was the partial tail of, while it holds it) may write the rest
  std::vector<int32_t> base_frozen, res_frozen;
  std::vector<int32_t> base_owner, res_owner;
  std::unordered_map<int32_t, Seq> seqs;
  int32_t next_id = 0;

  int32_t pop(bool base) {
    auto& st = base ? base_free : res_free;
    int32_t p = st.back();
    st.pop_back();
    (base ? base_ref : res_ref)[p] = 1;
    (base ? base_frozen : res_frozen)[p] = 0;
    (base ? base_owner : res_owner)[p] = -1;
    return p;
  }
  // seq drops its reference to page p
  void release(bool base, int32_t p, int32_t seq) {
    auto& own = base ? base_owner : res_owner;
    if (own[p] == seq) own[p] = -1;
    if (--(base ? base_ref : res_ref)[p] == 0) {
      (base ? base_free : res_free).push_back(p);
      (base ? base_frozen : res_frozen)[p] = 0;
      own[p] = -1;
    }
  }
  // seq may write rows >= row of its shared page p in place (its own frozen tail, past every
  // child's frozen rows)
  bool writes_in_place(bool base, int32_t p, int32_t seq, int32_t row) const {
    return (base ? base_owner : res_owner)[p] == seq && row >= (base ? base_frozen : res_frozen)[p];
  }
  Seq* find(int32_t id) {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
  const Seq* find(int32_t id) const {
    auto it = seqs.find(id);
    return it == seqs.end() ? nullptr : &it->second;
  }
};

extern "C" {

int32_t forkkv_alloc_create(int32_t num_base_pages, int32_t num_res_pages, int32_t page_size,
                            forkkv_alloc** out) {
  if (!out || num_base_pages < 0 || num_res_pages < 0) return FORKKV_ERR_INVALID_ARG;
  if (page_size != FORKKV_PAGE_SIZE) return FORKKV_ERR_UNSUPPORTED;
  forkkv_alloc* a = new (std::nothrow) forkkv_alloc();
  if (!a) return FORKKV_ERR_INVALID_ARG;
  try {
    a->base_free.resize(num_base_pages);
    a->res_free.resize(num_res_pages);
    for (int32_t i = 0; i < num_base_pages; ++i) a->base_free[i] = num_base_pages - 1 - i;
    for (int32_t i = 0; i < num_res_pages; ++i) a->res_free[i] = num_res_pages - 1 - i;
    a->base_ref.assign(num_base_pages, 0);
    a->res_ref.assign(num_res_pages, 0);
    a->base_frozen.assign(num_base_pages, 0);
    a->res_frozen.assign(num_res_pages, 0);
    a->base_owner.assign(num_base_pages, -1);
    a->res_owner.assign(num_res_pages, -1);
  } catch (...) {
    delete a;
    return FORKKV_ERR_INVALID_ARG;
  }
  *out = a;
  return FORKKV_OK;
}

int32_t forkkv_alloc_destroy(forkkv_alloc* alloc) {
  delete alloc;
  return FORKKV_OK;
}

int32_t forkkv_seq_create(forkkv_alloc* a, int32_t n_tokens, int32_t* seq_out) {
  if (!a || !seq_out || n_tokens < 0) return FORKKV_ERR_INVALID_ARG;
  const int32_t npg = ceil_div(n_tokens, a->page);
  if (npg > static_cast<int32_t>(a->base_free.size()) || npg > static_cast<int32_t>(a->res_free.size()))
    return FORKKV_ERR_OUT_OF_PAGES;
  try {
    Seq s;
    s.length = n_tokens;
    s.base.reserve(npg);
    s.res.reserve(npg);
    const int32_t id = a->next_id;
    a->seqs.emplace(id, Seq());  // may throw before any page moves
    for (int32_t i = 0; i < npg; ++i) s.base.push_back(a->pop(true));
    for (int32_t i = 0; i < npg; ++i) s.res.push_back(a->pop(false));
    a->seqs[id] = std::move(s);
    a->next_id++;
    *seq_out = id;
  } catch (...) {
    return FORKKV_ERR_INVALID_ARG;
  }
  return FORKKV_OK;
}

int32_t forkkv_fork(forkkv_alloc* a, int32_t parent, int32_t prefix_len, uint32_t flags,
                    int32_t* child_out, forkkv_cow_job* jobs, int32_t jobs_cap, int32_t* n_jobs) {
  if (!a || !child_out || !n_jobs || jobs_cap < 0 || (jobs_cap > 0 && !jobs)) return FORKKV_ERR_INVALID_ARG;
  if (flags & ~(FORKKV_FORK_SHARE_RES | FORKKV_FORK_FREEZE_TAIL)) return FORKKV_ERR_INVALID_ARG;
  const Seq* par = a->find(parent);
  if (!par || prefix_len < 0 || prefix_len > par->length) return FORKKV_ERR_INVALID_ARG;
  const bool share_res = (flags & FORKKV_FORK_SHARE_RES) != 0;
  const int32_t P = a->page;
  const bool inherit = par->hole_len && prefix_len > par->hole_start;  // the prefix spans the parent's hole
  const int32_t slot_end = par->slots_of(prefix_len);
  const int32_t nf = slot_end / P, t = slot_end % P;
  const int32_t npg = nf + (t ? 1 : 0);
  // freeze: only for an unaligned tail, and only if the child would not hold two holes
  const bool freeze = (flags & FORKKV_FORK_FREEZE_TAIL) && t && !inherit;
  // rows of the parent's tail page the parent has written (the rest may never have been)
  const int32_t written = freeze ? (par->slots() - nf * P < P ? par->slots() - nf * P : P) : P;
  int32_t need_base, need_res, nj;
  if (freeze) {
    need_base = 0;
    need_res = share_res ? 0 : npg;
    nj = (written < P ? 1 : 0) + (share_res ? (written < P ? 1 : 0) : 1);
  } else {
    need_base = t ? 1 : 0;
    need_res = share_res ? (t ? 1 : 0) : npg;
    nj = (t ? 1 : 0) * (share_res ? 2 : 1);
  }
  if (nj > jobs_cap) return FORKKV_ERR_INVALID_ARG;
  if (need_base > static_cast<int32_t>(a->base_free.size()) || need_res > static_cast<int32_t>(a->res_free.size()))
    return FORKKV_ERR_OUT_OF_PAGES;
  try {
    Seq c;
    c.length = prefix_len;
    c.base.reserve(npg);
    c.res.reserve(npg);
    const int32_t id = a->next_id;
    a->seqs.emplace(id, Seq());  // may throw (and invalidate nothing else) before any change
    par = a->find(parent);       // re-find: emplace may rehash
    int32_t k = 0;
    if (inherit) {
      c.hole_start = par->hole_start;
      c.hole_len = par->hole_len;
    }
    for (int32_t i = 0; i < nf; ++i) {
      c.base.push_back(par->base[i]);
      a->base_ref[par->base[i]]++;
    }
    if (freeze) {
      // the parent's tail page, read-only for the child: rows [0, t) are the prefix's; the
      // child's slots [slot_end, (nf + 1) P) are a hole, its own tokens start on a fresh page
      const int32_t tp = par->base[nf];
      c.base.push_back(tp);
      a->base_ref[tp]++;
      if (a->base_frozen[tp] < t) a->base_frozen[tp] = t;
      if (a->base_owner[tp] < 0 && par->slots() < (nf + 1) * P) a->base_owner[tp] = parent;
      if (written < P) jobs[k++] = forkkv_cow_job{tp, tp, written, FORKKV_JOB_BASE_ZERO};
      c.hole_start = slot_end;
      c.hole_len = P - t;
      if (share_res) {
        for (int32_t i = 0; i <= nf; ++i) {
          c.res.push_back(par->res[i]);
          a->res_ref[par->res[i]]++;
        }
        const int32_t rp = par->res[nf];
        if (a->res_frozen[rp] < t) a->res_frozen[rp] = t;
        if (a->res_owner[rp] < 0 && par->slots() < (nf + 1) * P) a->res_owner[rp] = parent;
        if (written < P) jobs[k++] = forkkv_cow_job{rp, rp, written, FORKKV_JOB_RES_ZERO};
      } else {
        for (int32_t i = 0; i < npg; ++i) c.res.push_back(a->pop(false));
        // the child's own residual rows of the hole are never written
        jobs[k++] = forkkv_cow_job{c.res[nf], c.res[nf], t, FORKKV_JOB_RES_ZERO};
      }
    } else {
      if (t) {
        const int32_t dst = a->pop(true);
        jobs[k++] = forkkv_cow_job{par->base[nf], dst, t, FORKKV_JOB_BASE};
        c.base.push_back(dst);
      }
      if (share_res) {
        for (int32_t i = 0; i < nf; ++i) {
          c.res.push_back(par->res[i]);
          a->res_ref[par->res[i]]++;
        }
        if (t) {
          const int32_t dst = a->pop(false);
          jobs[k++] = forkkv_cow_job{par->res[nf], dst, t, FORKKV_JOB_RES};
          c.res.push_back(dst);
        }
      } else {
        for (int32_t i = 0; i < npg; ++i) c.res.push_back(a->pop(false));
      }
    }
    a->seqs[id] = std::move(c);
    a->next_id++;
    *child_out = id;
    *n_jobs = k;
  } catch (...) {
    return FORKKV_ERR_INVALID_ARG;
  }
  return FORKKV_OK;
}

int32_t forkkv_append(forkkv_alloc* a, int32_t seq, int32_t n_tokens, forkkv_cow_job* jobs, int32_t jobs_cap,
                      int32_t* n_jobs) {
  if (!a || !n_jobs || n_tokens < 0 || jobs_cap < 0 || (jobs_cap > 0 && !jobs)) return FORKKV_ERR_INVALID_ARG;
  Seq* s = a->find(seq);
  if (!s) return FORKKV_ERR_INVALID_ARG;
  const int32_t P = a->page;
  const int64_t S = s->slots();
  if (S + n_tokens > INT32_MAX) return FORKKV_ERR_INVALID_ARG;
  const int32_t grow = ceil_div(S + n_tokens, P) - ceil_div(S, P);
  const int32_t tail = static_cast<int32_t>(S % P);
  // a shared partial last page is copied first, unless it is this sequence's frozen tail
  const bool cow_base = n_tokens > 0 && tail && a->base_ref[s->base.back()] > 1 &&
                        !a->writes_in_place(true, s->base.back(), seq, tail);
  const bool cow_res = n_tokens > 0 && tail && a->res_ref[s->res.back()] > 1 &&
                       !a->writes_in_place(false, s->res.back(), seq, tail);
  const int32_t nj = (cow_base ? 1 : 0) + (cow_res ? 1 : 0);
  if (nj > jobs_cap) return FORKKV_ERR_INVALID_ARG;
  if (grow + (cow_base ? 1 : 0) > static_cast<int32_t>(a->base_free.size()) ||
      grow + (cow_res ? 1 : 0) > static_cast<int32_t>(a->res_free.size()))
    return FORKKV_ERR_OUT_OF_PAGES;
  try {
    s->base.reserve(s->base.size() + grow);  // may throw before any change
    s->res.reserve(s->res.size() + grow);
  } catch (...) {
    return FORKKV_ERR_INVALID_ARG;
  }
  int32_t k = 0;
  if (cow_base) {
    const int32_t old = s->base.back();
    const int32_t dst = a->pop(true);
    a->release(true, old, seq);
    s->base.back() = dst;
    jobs[k++] = forkkv_cow_job{old, dst, tail, FORKKV_JOB_BASE};
  }
  for (int32_t i = 0; i < grow; ++i) s->base.push_back(a->pop(true));
  if (cow_res) {
    const int32_t old = s->res.back();
    const int32_t dst = a->pop(false);
    a->release(false, old, seq);
    s->res.back() = dst;
    jobs[k++] = forkkv_cow_job{old, dst, tail, FORKKV_JOB_RES};
  }
  for (int32_t i = 0; i < grow; ++i) s->res.push_back(a->pop(false));
  s->length = static_cast<int32_t>(s->length + n_tokens);
  *n_jobs = k;
  return FORKKV_OK;
}

int32_t forkkv_free(forkkv_alloc* a, int32_t seq) {
  if (!a) return FORKKV_ERR_INVALID_ARG;
  Seq* s = a->find(seq);
  if (!s) return FORKKV_ERR_INVALID_ARG;
  for (int32_t p : s->base)
    if (a->base_ref[p] <= 0) return FORKKV_ERR_REFCOUNT;
  for (int32_t p : s->res)
    if (a->res_ref[p] <= 0) return FORKKV_ERR_REFCOUNT;
  // pushes never exceed the pool size, so reserve once to keep push_back from throwing
  a->base_free.reserve(a->base_ref.size());
  a->res_free.reserve(a->res_ref.size());
  for (int32_t p : s->base) a->release(true, p, seq);
  for (int32_t p : s->res) a->release(false, p, seq);
  a->seqs.erase(seq);
  return FORKKV_OK;
}

int32_t forkkv_abort(forkkv_alloc* a, int32_t seq, int32_t* n_base_released, int32_t* n_res_released) {
  if (!a) return FORKKV_ERR_INVALID_ARG;
  const Seq* s = a->find(seq);
  if (!s) return FORKKV_ERR_INVALID_ARG;
  int32_t nb = 0, nr = 0;
  for (int32_t p : s->base) nb += a->base_ref[p] == 1;
  for (int32_t p : s->res) nr += a->res_ref[p] == 1;
  const int32_t rc = forkkv_free(a, seq);
  if (rc != FORKKV_OK) return rc;
  if (n_base_released) *n_base_released = nb;
  if (n_res_released) *n_res_released = nr;
  return FORKKV_OK;
}

int32_t forkkv_commit(forkkv_alloc* a, int32_t seq, int32_t lcp_len, const int32_t* siblings, int32_t n_siblings,
                      forkkv_cow_job* jobs, int32_t jobs_cap, int32_t* n_jobs) {
  if (!a || !n_jobs || n_siblings < 0 || (n_siblings > 0 && !siblings) || jobs_cap < 0 || (jobs_cap > 0 && !jobs))
    return FORKKV_ERR_INVALID_ARG;
  Seq* s = a->find(seq);
  if (!s || lcp_len < 0 || lcp_len > s->length) return FORKKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_siblings; ++i) {
    if (siblings[i] == seq || !a->find(siblings[i])) return FORKKV_ERR_INVALID_ARG;
    for (int32_t k = 0; k < i; ++k)
      if (siblings[k] == siblings[i]) return FORKKV_ERR_INVALID_ARG;
  }
  const int32_t P = a->page;
  const int32_t new_slots = s->slots_of(lcp_len);  // the hole goes too if the prefix ends at or before it
  const int32_t keep = ceil_div(new_slots, P), t = new_slots % P;
  const int32_t np = static_cast<int32_t>(s->base.size());
  // Everything is decided before anything changes: the decrements that the sibling frees and the
  // truncation will make (a page appears at most once in one sequence), the pages they release,
  // and whether the boundary page is still shared afterwards.
  std::unordered_map<int32_t, int32_t> dec_b, dec_r;
  try {
    for (int32_t i = 0; i < n_siblings; ++i) {
      const Seq* o = a->find(siblings[i]);
      for (int32_t p : o->base) dec_b[p]++;
      for (int32_t p : o->res) dec_r[p]++;
    }
    for (int32_t j = keep; j < np; ++j) {
      dec_b[s->base[j]]++;
      dec_r[s->res[j]]++;
    }
  } catch (...) {
    return FORKKV_ERR_INVALID_ARG;
  }
  int32_t free_b = static_cast<int32_t>(a->base_free.size()), free_r = static_cast<int32_t>(a->res_free.size());
  for (const auto& e : dec_b) {
    if (a->base_ref[e.first] < e.second) return FORKKV_ERR_REFCOUNT;
    free_b += a->base_ref[e.first] == e.second;
  }
  for (const auto& e : dec_r) {
    if (a->res_ref[e.first] < e.second) return FORKKV_ERR_REFCOUNT;
    free_r += a->res_ref[e.first] == e.second;
  }
  auto after = [](const std::vector<int32_t>& ref, const std::unordered_map<int32_t, int32_t>& dec, int32_t p) {
    auto it = dec.find(p);
    return ref[p] - (it == dec.end() ? 0 : it->second);
  };
  // a boundary page still shared is split unless it is this sequence's own frozen tail and the
  // rows it will write lie past every child's frozen rows (a sibling that owned it is gone by then)
  const bool split_b = t != 0 && after(a->base_ref, dec_b, s->base[keep - 1]) > 1 &&
                       !a->writes_in_place(true, s->base[keep - 1], seq, t);
  const bool split_r = t != 0 && after(a->res_ref, dec_r, s->res[keep - 1]) > 1 &&
                       !a->writes_in_place(false, s->res[keep - 1], seq, t);
  if ((split_b ? 1 : 0) + (split_r ? 1 : 0) > jobs_cap) return FORKKV_ERR_INVALID_ARG;
  if ((split_b && free_b < 1) || (split_r && free_r < 1)) return FORKKV_ERR_OUT_OF_PAGES;
  // 1. abort the siblings, in the order given
  for (int32_t i = 0; i < n_siblings; ++i)
    if (forkkv_free(a, siblings[i]) != FORKKV_OK) return FORKKV_ERR_REFCOUNT;  // excluded by the checks above
  s = a->find(seq);
  // 2. truncate: pages past the committed prefix, base then residual, in logical order
  a->base_free.reserve(a->base_ref.size());
  a->res_free.reserve(a->res_ref.size());
  for (int32_t j = keep; j < np; ++j) a->release(true, s->base[j], seq);
  for (int32_t j = keep; j < np; ++j) a->release(false, s->res[j], seq);
  s->base.resize(keep);
  s->res.resize(keep);
  // 3. a boundary page still shared is split: a private copy of its first t rows
  int32_t k = 0;
  if (split_b) {
    const int32_t old = s->base[keep - 1], dst = a->pop(true);
    a->release(true, old, seq);
    s->base[keep - 1] = dst;
    jobs[k++] = forkkv_cow_job{old, dst, t, FORKKV_JOB_BASE};
  }
  if (split_r) {
    const int32_t old = s->res[keep - 1], dst = a->pop(false);
    a->release(false, old, seq);
    s->res[keep - 1] = dst;
    jobs[k++] = forkkv_cow_job{old, dst, t, FORKKV_JOB_RES};
  }
  if (s->hole_len && lcp_len <= s->hole_start) s->hole_start = s->hole_len = 0;
  s->length = lcp_len;
  *n_jobs = k;
  return FORKKV_OK;
}

int32_t forkkv_lcp_len(const int32_t* spec, int32_t n_spec, const int32_t* observed, int32_t n_observed,
                       int32_t* out) {
  if (!out || n_spec < 0 || n_observed < 0 || (n_spec > 0 && !spec) || (n_observed > 0 && !observed))
    return FORKKV_ERR_INVALID_ARG;
  int32_t n = 0;
  const int32_t m = n_spec < n_observed ? n_spec : n_observed;
  while (n < m && spec[n] == observed[n]) ++n;
  *out = n;
  return FORKKV_OK;
}

int32_t forkkv_seq_len(const forkkv_alloc* a, int32_t seq, int32_t* len_out) {
  if (!a || !len_out) return FORKKV_ERR_INVALID_ARG;
  const Seq* s = a->find(seq);
  if (!s) return FORKKV_ERR_INVALID_ARG;
  *len_out = s->length;
  return FORKKV_OK;
}

int32_t forkkv_page_tables(const forkkv_alloc* a, const int32_t* seqs, int32_t n, int32_t stride, int32_t* bpt,
                           int32_t* rpt, int32_t* seq_lens) {
  if (!a || n < 0 || stride < 0 || (n > 0 && (!seqs || !bpt || !rpt || !seq_lens))) return FORKKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const Seq* s = a->find(seqs[i]);
    if (!s || static_cast<int64_t>(s->base.size()) > stride) return FORKKV_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    const Seq* s = a->find(seqs[i]);
    int32_t* b = bpt + static_cast<int64_t>(i) * stride;
    int32_t* r = rpt + static_cast<int64_t>(i) * stride;
    const int32_t np = static_cast<int32_t>(s->base.size());
    for (int32_t j = 0; j < stride; ++j) {
      b[j] = j < np ? s->base[j] : -1;
      r[j] = j < np ? s->res[j] : -1;
    }
    seq_lens[i] = s->slots();
  }
  return FORKKV_OK;
}

int32_t forkkv_slot_maps(const forkkv_alloc* a, const int32_t* seqs, int32_t n, int32_t* holes) {
  if (!a || n < 0 || (n > 0 && (!seqs || !holes))) return FORKKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (!a->find(seqs[i])) return FORKKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const Seq* s = a->find(seqs[i]);
    holes[2 * i] = s->hole_start;
    holes[2 * i + 1] = s->hole_len;
  }
  return FORKKV_OK;
}

int32_t forkkv_refcount(const forkkv_alloc* a, int32_t kind, int32_t page, int32_t* out) {
  if (!a || !out || (kind != FORKKV_JOB_BASE && kind != FORKKV_JOB_RES)) return FORKKV_ERR_INVALID_ARG;
  const auto& rf = kind == FORKKV_JOB_BASE ? a->base_ref : a->res_ref;
  if (page < 0 || page >= static_cast<int32_t>(rf.size())) return FORKKV_ERR_BAD_PAGE;
  *out = rf[page];
  return FORKKV_OK;
}

int32_t forkkv_stats_get(const forkkv_alloc* a, forkkv_stats* out) {
  if (!a || !out) return FORKKV_ERR_INVALID_ARG;
  forkkv_stats s{};
  s.n_seqs = static_cast<int32_t>(a->seqs.size());
  for (int32_t c : a->base_ref) {
    s.base_live += c > 0;
    s.base_shared += c > 1;
    s.base_refsum += c;
  }
  for (int32_t c : a->res_ref) {
    s.res_live += c > 0;
    s.res_shared += c > 1;
    s.res_refsum += c;
  }
  s.base_free = static_cast<int32_t>(a->base_free.size());
  s.res_free = static_cast<int32_t>(a->res_free.size());
  *out = s;
  return FORKKV_OK;
}

}  // extern "C"
