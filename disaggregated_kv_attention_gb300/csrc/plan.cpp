// Decode work planning: fork-tree segments -> work items.
//
// Agents forked from one trunk alias the same base pages (ForkKV L2 section 3,
// Figure 6; ForkServe "Methods", CoW tree).  Reading such a page once for
// every agent that maps it is what makes sharing pay in HBM bytes, so the plan
// groups, per run of logical pages, the agents whose page tables hold the same
// physical base page there.  The groups fall out of the page tables alone: walk
// the logical page index, and split a group of agents whenever their physical
// pages differ (or some of them end).  Each segment (agent group, page range)
// is then cut into items of at most 4 agents and a bounded number of 128-key
// blocks (8 pages).
#include <algorithm>
#include <array>
#include <climits>
#include <cstdint>
#include <functional>
#include <map>
#include <queue>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/forkkv.h"

namespace {

// SMs of the current device (one persistent decode CTA each); 152 (a GB300) when no device
// answers, e.g. when a plan is built on a host without a GPU.
int32_t device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();  // leave no sticky error behind for the caller
    return 152;
  }
  return n;
}

struct Segment {
  std::vector<int32_t> agents;
  int32_t p0, p1;
};

// Pages per pipeline stage of the decode kernel: one 128-key block, whatever the
// group size (the block's base tiles are read once and reused by every agent).
constexpr int32_t kStagePages = 8;
constexpr int32_t kMaxGroup = 4;
int32_t pages_per_stage(int32_t) { return kStagePages; }

int32_t plan_build(const int32_t* bpt, const int32_t* seq_lens, int32_t n_agents, int32_t pt_stride,
                   int32_t num_kv_heads, int32_t target_ctas, int32_t* plan, int32_t plan_cap_ints,
                   forkkv_plan_info* info) {
  if (!bpt || !seq_lens || !info || n_agents < 1 || pt_stride < 1 || num_kv_heads < 1 || target_ctas < 0)
    return FORKKV_ERR_INVALID_ARG;
  if (target_ctas == 0) target_ctas = device_sms();  // one persistent CTA per SM
  std::vector<int32_t> npages(n_agents);
  for (int32_t a = 0; a < n_agents; ++a) {
    if (seq_lens[a] < 1) return FORKKV_ERR_INVALID_ARG;
    npages[a] = (seq_lens[a] + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE;
    if (npages[a] > pt_stride) return FORKKV_ERR_INVALID_ARG;
    for (int32_t j = 0; j < npages[a]; ++j)
      if (bpt[(int64_t)a * pt_stride + j] < 0) return FORKKV_ERR_BAD_PAGE;
  }

  // 1. segments of the fork tree, by an explicit-stack walk over logical pages
  std::vector<Segment> segs;
  struct Frame {
    std::vector<int32_t> group;
    int32_t i0;
  };
  std::vector<Frame> stack;
  {
    std::vector<int32_t> all(n_agents);
    for (int32_t a = 0; a < n_agents; ++a) all[a] = a;
    stack.push_back({all, 0});
  }
  while (!stack.empty()) {
    Frame f = std::move(stack.back());
    stack.pop_back();
    int32_t i = f.i0;
    for (;;) {
      bool same = true;
      const int32_t a0 = f.group[0];
      for (int32_t a : f.group) {
        if (i >= npages[a] || bpt[(int64_t)a * pt_stride + i] != bpt[(int64_t)a0 * pt_stride + i]) {
          same = false;
          break;
        }
      }
      if (!same) break;
      ++i;
    }
    if (i > f.i0) segs.push_back({f.group, f.i0, i});
    // agents still active at page i, grouped by their physical page (first-seen order)
    std::vector<int32_t> order;
    std::map<int32_t, std::vector<int32_t>> cls;
    for (int32_t a : f.group) {
      if (i >= npages[a]) continue;
      const int32_t pg = bpt[(int64_t)a * pt_stride + i];
      if (!cls.count(pg)) order.push_back(pg);
      cls[pg].push_back(a);
    }
    for (auto it = order.rbegin(); it != order.rend(); ++it) stack.push_back({cls[*it], i});
  }

  // 2. groups of at most 4 agents (4, then 2, 1 for the remainder)
  struct Chunk {
    int32_t agents[8];
    int32_t na, p0, p1, stages, seg, grp;  // grp: the chunk's index among its segment's groups
  };
  std::vector<Chunk> chunks;
  for (size_t si = 0; si < segs.size(); ++si) {
    const Segment& s = segs[si];
    size_t k = 0;
    int32_t grp = 0;
    while (k < s.agents.size()) {
      const size_t left = s.agents.size() - k;
      const int32_t na = left >= kMaxGroup ? kMaxGroup : left >= 2 ? 2 : 1;
      Chunk c{};
      for (int32_t x = 0; x < 8; ++x) c.agents[x] = x < na ? s.agents[k + x] : -1;
      c.na = na;
      c.p0 = s.p0;
      c.p1 = s.p1;
      const int32_t wpp = pages_per_stage(na);
      c.stages = (s.p1 - s.p0 + wpp - 1) / wpp;
      c.seg = (int32_t)si;
      c.grp = grp++;
      chunks.push_back(c);
      k += na;
    }
  }

  // 3. a stage cap per group size (chunks are cut into near-equal items of at most that many
  //    blocks) and a spread of the (item, head) units over the CTAs.  A unit's cost is its
  //    time on one SM as measured for the decode kernel on a GB300 (ns): a block takes about
  //    930 per agent, and no less than 2400 however few agents share it (the copies and the
  //    value products of a block then set the pace); starting a unit and writing its
  //    partials add about 3000.  Units go largest first to the least loaded CTA (LPT).  The
  //    caps are chosen by coordinate descent on the makespan, each from the longest chunk
  //    down, keeping the larger cap on ties (fewer partials to merge).
  const int32_t C_max = target_ctas;
  auto gi = [](int32_t na) { return na >= 4 ? 2 : na - 1; };  // group-size class of a chunk
  int32_t max_stages[3] = {1, 1, 1};
  bool present[3] = {false, false, false};
  for (const Chunk& c : chunks) {
    max_stages[gi(c.na)] = std::max(max_stages[gi(c.na)], c.stages);
    present[gi(c.na)] = true;
  }
  auto unit_cost = [](int32_t blocks, int32_t na) {
    return (int64_t)blocks * std::max<int64_t>(930 * (int64_t)na, 2400) + 3000;
  };
  struct Unit {
    int64_t cost;
    int32_t code;
    int32_t seg, first, head, grp;  // siblings: the groups of one segment on the same pages and head
  };
  // items under caps T: (chunk index, first stage, end stage)
  auto make_items = [&](const int32_t* T, std::vector<std::array<int32_t, 3>>& out) {
    out.clear();
    for (size_t ci = 0; ci < chunks.size(); ++ci) {
      const Chunk& c = chunks[ci];
      const int32_t t = T[gi(c.na)];
      const int32_t parts = (c.stages + t - 1) / t;
      for (int32_t k = 0; k < parts; ++k)
        out.push_back({(int32_t)ci, (int32_t)((int64_t)c.stages * k / parts),
                       (int32_t)((int64_t)c.stages * (k + 1) / parts)});
    }
  };
  auto count_items = [&](const int32_t* T) {
    int64_t n = 0;
    for (const Chunk& c : chunks) n += (c.stages + T[gi(c.na)] - 1) / T[gi(c.na)];
    return n;
  };
  // LPT spread of the units of `its` over at most C_max CTAs; returns the makespan
  auto spread = [&](const std::vector<std::array<int32_t, 3>>& its, std::vector<std::vector<int32_t>>* lists) {
    std::vector<Unit> units;
    units.reserve(its.size() * num_kv_heads);
    for (size_t i = 0; i < its.size(); ++i) {
      const Chunk& c = chunks[its[i][0]];
      const int64_t cost = unit_cost(its[i][2] - its[i][1], c.na);
      for (int32_t h = 0; h < num_kv_heads; ++h)
        units.push_back({cost, (int32_t)(i * num_kv_heads + h), c.seg, its[i][1], h, c.grp});
    }
    // Largest first; among equal costs, the groups that share a segment's pages (a trunk read by
    // several agent groups) next to each other for the same pages and head, so that they land on
    // CTAs of equal load and stream those pages at the same time: the repeats then come from L2.
    std::stable_sort(units.begin(), units.end(), [](const Unit& x, const Unit& y) {
      if (x.cost != y.cost) return x.cost > y.cost;
      if (x.seg != y.seg) return x.seg < y.seg;
      if (x.first != y.first) return x.first < y.first;
      if (x.head != y.head) return x.head < y.head;
      return x.grp < y.grp;
    });
    const int32_t C = (int32_t)std::min<int64_t>(C_max, (int64_t)units.size());
    using Load = std::pair<int64_t, int32_t>;  // (load, CTA): the least loaded, then the lowest index
    std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
    for (int32_t c = 0; c < C; ++c) heap.push({0, c});
    if (lists) lists->assign(C, {});
    int64_t makespan = 0;
    for (const Unit& u : units) {
      Load l = heap.top();
      heap.pop();
      l.first += u.cost;
      makespan = std::max(makespan, l.first);
      if (lists) (*lists)[l.second].push_back(u.code);
      heap.push(l);
    }
    return makespan;
  };
  std::vector<std::array<int32_t, 3>> its;
  int32_t T[3] = {max_stages[0], max_stages[1], max_stages[2]};
  make_items(T, its);
  int64_t best = spread(its, nullptr);
  for (int round = 0; round < 2; ++round) {
    for (int g = 0; g < 3; ++g) {
      if (!present[g]) continue;
      int32_t trial[3] = {T[0], T[1], T[2]};
      int64_t last_count = -1;
      for (int32_t t = max_stages[g]; t >= 1; --t) {
        trial[g] = t;
        const int64_t count = count_items(trial);
        if (count == last_count) continue;  // the same items as the previous cap
        last_count = count;
        if (count * num_kv_heads > 16 * (int64_t)C_max) break;  // at most 16 units per CTA
        make_items(trial, its);
        const int64_t m = spread(its, nullptr);
        if (m < best) {
          best = m;
          T[g] = t;
        }
      }
    }
  }
  make_items(T, its);
  std::vector<std::vector<int32_t>> lists;
  spread(its, &lists);

  // 4. items, slots, the per-agent slot lists and the CTAs' unit lists
  std::vector<int32_t> items;
  std::vector<std::vector<int32_t>> agent_slots(n_agents);
  int32_t n_items = 0, n_slots = 0;
  for (const auto& itm : its) {
    const Chunk& c = chunks[itm[0]];
    const int32_t wpp = pages_per_stage(c.na);
    const int32_t p0 = c.p0 + itm[1] * wpp, p1 = std::min(c.p1, c.p0 + itm[2] * wpp);
    int32_t rec[FORKKV_PLAN_ITEM_INTS] = {0};
    rec[0] = p0;
    rec[1] = p1;
    rec[2] = c.na;
    rec[3] = wpp;
    for (int32_t x = 0; x < 8; ++x) rec[4 + x] = x < c.na ? c.agents[x] : c.agents[0];
    rec[12] = n_slots;
    items.insert(items.end(), rec, rec + FORKKV_PLAN_ITEM_INTS);
    for (int32_t x = 0; x < c.na; ++x) agent_slots[c.agents[x]].push_back(n_slots + x);
    n_slots += c.na;
    ++n_items;
  }
  const int32_t n_ctas = (int32_t)lists.size();
  const int64_t n_units = (int64_t)n_items * num_kv_heads;
  const int64_t need = (int64_t)items.size() + n_agents + 1 + n_slots + n_units * FORKKV_PLAN_UNIT_INTS;
  if (need > INT32_MAX) return FORKKV_ERR_INVALID_ARG;
  info->n_items = n_items;
  info->n_slots = n_slots;
  info->n_ctas = n_ctas;
  info->n_units = (int32_t)n_units;
  info->plan_ints = (int32_t)need;
  if (!plan) return FORKKV_OK;  // size query
  if (need > plan_cap_ints) return FORKKV_ERR_INVALID_ARG;
  std::copy(items.begin(), items.end(), plan);
  int32_t* off = plan + items.size();
  int32_t* sl = off + n_agents + 1;
  int32_t k = 0;
  for (int32_t a = 0; a < n_agents; ++a) {
    off[a] = k;
    for (int32_t s : agent_slots[a]) sl[k++] = s;
  }
  off[n_agents] = k;
  // unit records: CTA c starts at record c, its later units follow from n_ctas on, each
  // record naming the next one of its CTA
  int32_t* units = sl + n_slots;
  std::fill(units, units + n_units * FORKKV_PLAN_UNIT_INTS, 0);
  int32_t later = n_ctas;
  for (int32_t c = 0; c < n_ctas; ++c) {
    int32_t r = c;
    for (size_t j = 0; j < lists[c].size(); ++j) {
      const int32_t code = lists[c][j];
      const int32_t* it = &items[(size_t)(code / num_kv_heads) * FORKKV_PLAN_ITEM_INTS];
      int32_t* u = units + (int64_t)r * FORKKV_PLAN_UNIT_INTS;
      const int32_t next = j + 1 < lists[c].size() ? later++ : -1;
      u[0] = it[0];                   // first logical page
      u[1] = it[1];                   // end logical page
      u[2] = it[2];                   // agents in the group
      u[3] = code % num_kv_heads;     // KV head
      u[4] = it[12];                  // first partial slot
      u[5] = next;                    // the CTA's next unit
      for (int32_t x = 0; x < kMaxGroup; ++x) u[6 + x] = it[4 + x];
      r = next;
    }
  }
  return FORKKV_OK;
}

}  // namespace

extern "C" int32_t forkkv_plan_build(const int32_t* bpt, const int32_t* seq_lens, int32_t n_agents, int32_t pt_stride,
                                     int32_t num_kv_heads, int32_t target_ctas, int32_t* plan, int32_t plan_cap_ints,
                                     forkkv_plan_info* info) {
  try {
    return plan_build(bpt, seq_lens, n_agents, pt_stride, num_kv_heads, target_ctas, plan, plan_cap_ints, info);
  } catch (...) {
    return FORKKV_ERR_INVALID_ARG;
  }
}
