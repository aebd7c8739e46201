// ResidualAttention decode for sm_103a on the fifth-generation tensor cores.
//
// Restates ForkKV L2 sections 4 and 7 (deferred RoPE, associativity of the
// value path, dual-accumulator online softmax) as a split-KV decode:
//
//   split kernel  persistent: each CTA works through a list of units back to
//                 back.  A unit is (work item, KV head); a work item is a run of
//                 logical pages shared by up to 4 agents (a trunk of the fork
//                 tree) or one agent's own pages, walked in 128-key blocks.  With
//                 a plan the lists come from the host planner (balanced by cost);
//                 without one the units are dealt round-robin.  Buffer rings and
//                 barrier phases run on across units.
//     warp 0      producer: each block's base K and V tiles (read ONCE for the
//                 whole agent group) into two K and two V buffers, released
//                 separately, each agent's residual k/v tiles into a 4-slot ring;
//                 1-D bulk async copies, one per run of consecutive page ids,
//                 completing on mbarriers
//     warp 1      allocates tensor memory; stages B_k of the unit's head and one
//                 lane issues, per (block, agent):
//                   U    = Kr . B_k                 [128 keys x 128]  smem x smem
//     warp 15     stages Q of the unit's agents and issues, per (block, agent):
//                   S    = K . Q^T                  [128 keys x 16]   K from TMEM
//                 (K and S in rings of three in tensor memory)
//     warps 2..9  RoPE group, one key per thread and half of the columns per
//                 warp: K = Kb + RoPE_j(U), the rotation of the (small) residual
//                 term in bf16x2 and one rounding of K, written to tensor memory
//                 as the A operand of the score product
//     warps 10..13 softmax group, one key per thread: scores, length mask, block
//                 maxima across the group, lazy rescale of O (only when the
//                 running maximum grows by 2^8), P^T to shared memory; at the end
//                 of a unit one partial (m, l, acc, acc_r) per (agent, KV head)
//     warp 14     one lane issues, per block and for all its agents at once,
//                   O^T += Vb^T . P^T  and  R += Vr^T . P^T (rank-16 value path)
//                 and l as the product of a tile of ones with P^T.
//   combine       one CTA per (agent, KV head, query head): log-sum-exp merge of
//                 the partials, then out = (acc + acc_r . B_v[:, hD:(h+1)D]) / l,
//                 B_v applied once per query head.
// Every wait is on an mbarrier with a bounded spin; a timeout sets the device
// status word instead of hanging.
#include <math.h>

#include <algorithm>

#include "../internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fkv {
namespace {

constexpr int kMaxGroup = 4;                 // agents per work unit
constexpr int kBlockPages = 8;               // 128 keys per block
constexpr int kRopeWarps = 8;                // two per TMEM lane quadrant
constexpr int kSoftWarp0 = 2 + kRopeWarps;   // first of the four softmax warps
constexpr int kValueWarp = kSoftWarp0 + 4;   // issues the value products of each block
constexpr int kScoreWarp = kValueWarp + 1;   // issues the score products
constexpr int kThreads = (kScoreWarp + 1) * 32;
constexpr int kPartCols = kHeadDim + kRank;  // 144 floats per (slot, head, query head)
constexpr int kResSlots = 4;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kBlockTiles = kBlockPages * kBaseTile;         // 32 KB: one block of K (or V) tiles
constexpr int kOffK = 2048;                                  // 2 x K block (after barriers and state)
constexpr int kOffV = kOffK + 2 * kBlockTiles;               // 2 x V block
constexpr int kResSlotBytes = kBlockPages * kResTile;        // 4 KB: one agent's residual tiles of a block
// v_res of a block: two groups (block parity) of 5 units of 4 KB, units 0..3 for up to four
// agents and unit 4 a constant tile of ones.  Agent a of a block of na agents sits in
// unit 4 - na + a, so the agents and then the ones are consecutive 16-row atoms of the
// residual-value product's A operand.
constexpr int kVrGroupBytes = 5 * kResSlotBytes;
constexpr int kOffVr = kOffV + 2 * kBlockTiles;              // 2 x [4 x v_res | ones]
constexpr int kOffKr = kOffVr + 2 * kVrGroupBytes;           // 4 x k_res slot
constexpr int kOffQ = kOffKr + kResSlots * kResSlotBytes;    // 4 agents x 2 halves x Q^T [8 rows][128 B]
constexpr int kOffQZero = kOffQ + kMaxGroup * 2048;          // 1 KB of zeros: query-head rows 8..15
constexpr int kOffBk = kOffQZero + 1024;                     // 4 x B_k [16 ranks][128 d], base-tile layout
constexpr int kOffP = kOffBk + kMaxGroup * 4096;             // 2 x P^T [2 atoms (agents 0-1, 2-3)][128 keys][32 B]
constexpr int kSmemBytes = kOffP + 2 * 8192;                 // the dynamic window is 1024-byte aligned (checked)
// The residual-value product reads 8 atoms from the block's first agent on; the atoms past
// the ones tile (rows of the product that are never read) must lie inside the allocation.
static_assert(kOffVr + kVrGroupBytes + 3 * kResSlotBytes + 8 * kResSlotBytes <= kSmemBytes,
              "value-product atoms leave the allocation");
static_assert(kSmemBytes <= 227 * 1024, "more shared memory than a CTA may have");

// tensor memory columns: U (fp32, read out early in a step, so one buffer), K (bf16 pairs)
// and S in rings of 3, O^T [128 d x 8 agents' query heads] and the residual-value product
constexpr int kRing = 3;
constexpr uint32_t kTmU = 0, kTmKF = 128, kTmS = kTmKF + 64 * kRing, kTmO = 384, kTmR = 416, kTmCols = 512;
static_assert(kTmS + 16 * kRing <= kTmO, "tensor memory regions overlap");

enum {
  kKFull0, kKFull1, kVFull0, kVFull1, kKEmpty0, kKEmpty1, kVEmpty0, kVEmpty1,
  kKrFull0, kKrFull1, kKrFull2, kKrFull3, kKrEmpty0, kKrEmpty1, kKrEmpty2, kKrEmpty3,
  kUFull, kUFree, kKFFull0, kKFFull1, kKFFull2, kKFFree0, kKFFree1, kKFFree2, kSFull0, kSFull1, kSFull2,
  kSFree0, kSFree1, kSFree2,
  kPFull0, kPFull1, kPFree0, kPFree1, kRed0, kRed1, kODone0, kODone1, kUUnit, kSUnit, kEpiDone,
  kMmaDone, kValDone, kSDone, kNumBars
};
static_assert(kNumBars * 8 <= 384, "barriers overlap the state that follows them");

struct DecodeArgs {
  const uint8_t* k_base;
  const uint8_t* v_base;
  const uint8_t* k_res;
  const uint8_t* v_res;
  int32_t num_base_pages, num_res_pages, hkv, G;
  const __nv_bfloat16* q;  // [A][Hq][128]
  const int32_t* bpt;
  const int32_t* rpt;
  int32_t pt_stride;
  const int32_t* seq_lens;
  const int32_t* positions;
  const __nv_bfloat16* B_k;  // [n_adapters][16][Hkv*128]
  const int32_t* adapter_ids;
  int32_t n_adapters;
  const uint8_t* rope;
  int32_t rope_positions;
  float scale_log2;
  const int32_t* plan;     // items (FORKKV_PLAN_ITEM_INTS each), or null: one item per (agent, chunk)
  const int32_t* cta_off;  // plan mode: [n_ctas + 1] into units
  const int32_t* units;    // plan mode: item * hkv + head, grouped by CTA
  int32_t n_items, n_ctas;
  int32_t chunk_pages, chunks;
  int32_t n_agents, max_seq_len, n_slots;
  float* part;
  float* ml;
  uint32_t* status;
};

// One unit of work: an item (a page range walked by a group of agents) for one KV head.
struct Unit {
  int32_t p0, p1, na, slot_base, h;
  int32_t agents[kMaxGroup];
  __device__ __forceinline__ int blocks() const { return (p1 - p0 + kBlockPages - 1) / kBlockPages; }
  __device__ __forceinline__ int32_t agent(int x) const {
    int32_t r = agents[0];
#pragma unroll
    for (int i = 1; i < kMaxGroup; ++i)
      if (x == i) r = agents[i];
    return r;
  }
};

// Units of this CTA: [*first, *first + *count) of the plan's unit list, or every gridDim.x-th
// (agent chunk, head) pair without a plan.
__device__ __forceinline__ void cta_units(const DecodeArgs& a, int& first, int& count) {
  if (a.plan) {
    first = a.cta_off[blockIdx.x];
    count = a.cta_off[blockIdx.x + 1] - first;
    if (first < 0 || count < 0 || first + count > a.cta_off[a.n_ctas]) {
      flag_status(a.status, kDevBadArg);
      first = count = 0;
    }
  } else {
    const int total = a.n_items * a.hkv;
    first = blockIdx.x;
    count = blockIdx.x < total ? (total - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  }
}

__device__ __forceinline__ Unit load_unit(const DecodeArgs& a, int first, int k) {
  Unit u;
  int32_t item, head;
  if (a.plan) {
    const int32_t code = a.units[first + k];
    item = code / a.hkv;
    head = code - item * a.hkv;
  } else {
    const int32_t code = first + k * gridDim.x;
    item = code / a.hkv;
    head = code - item * a.hkv;
  }
  u.h = head;
  if (a.plan) {
    if ((uint32_t)item >= (uint32_t)a.n_items) {
      flag_status(a.status, kDevBadArg);
      item = 0;
    }
    const int32_t* p = a.plan + (int64_t)item * FORKKV_PLAN_ITEM_INTS;
    u.p0 = p[0];
    u.p1 = p[1];
    u.na = p[2];
#pragma unroll
    for (int i = 0; i < kMaxGroup; ++i) u.agents[i] = p[4 + i];
    u.slot_base = p[12];
    if (u.na != 1 && u.na != 2 && u.na != 4) {  // the value products stack the slots of 1, 2 or 4 agents
      flag_status(a.status, kDevBadArg);
      u.na = 1;
      u.p1 = u.p0;
    }
    if (u.slot_base < 0 || u.slot_base + u.na > a.n_slots) {
      flag_status(a.status, kDevBadArg);
      u.p1 = u.p0;  // empty: reads nothing, writes nothing
      u.slot_base = -1;
    }
  } else {
    const int32_t agent = item / a.chunks, c = item % a.chunks;
    const int32_t L = min(a.seq_lens[agent], a.max_seq_len);
    const int32_t npg = (L + kPage - 1) / kPage;
    u.p0 = c * a.chunk_pages;
    u.p1 = min(u.p0 + a.chunk_pages, npg);
    u.na = 1;
#pragma unroll
    for (int i = 0; i < kMaxGroup; ++i) u.agents[i] = agent;
    u.slot_base = item;
  }
  if ((uint32_t)u.h >= (uint32_t)a.hkv) {
    flag_status(a.status, kDevBadArg);
    u.h = 0;
    u.p1 = u.p0;
  }
#pragma unroll
  for (int i = 0; i < kMaxGroup; ++i)
    if ((uint32_t)u.agents[i] >= (uint32_t)a.n_agents) {
      flag_status(a.status, kDevBadArg);
      u.agents[i] = 0;
      u.p1 = u.p0;
    }
  if (u.p0 < 0 || u.p1 > a.pt_stride) {
    flag_status(a.status, kDevBadArg);
    u.p0 = u.p1 = 0;
  }
  if (u.p1 < u.p0) u.p1 = u.p0;
  return u;
}

// Lanes work in groups of 8: an active group copies the nvp (<= 8) page tiles of a block,
// whose ids sit in its lanes 8 q + p, into consecutive tiles at `dst` (the group's own
// destination), raising the byte count `bar` expects (the caller arrives).  Consecutive
// ids go as one bulk copy from the group's first lane, otherwise every lane copies its
// own page, so the groups of a warp issue side by side.  When rows < 16 only the first
// rows of the last page are copied and the rest of that tile is zeroed first (rows past
// every sequence may never have been written, and a zero probability must not meet a
// NaN).  A base tile keeps its rows in two 2048-byte halves (128 bytes a row), a residual
// tile in one (32 bytes a row).
__device__ __forceinline__ void copy_group(const uint8_t* pool, bool base, int32_t id, int nvp, int rows, uint8_t* dst,
                                          uint64_t* bar, bool active, int lane) {
  const int p = lane & 7;
  const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
  const int full = rows < kPage ? nvp - 1 : nvp;  // pages copied whole
  if (active && full < nvp) {
    uint8_t* t = dst + full * tile;
    const uint32_t keep = rows * rb, half = base ? 2048u : tile;  // bytes kept per half
    for (uint32_t o = keep + 16 * p; o < half; o += 16 * 8) {
      *reinterpret_cast<uint4*>(t + o) = make_uint4(0u, 0u, 0u, 0u);
      if (base) *reinterpret_cast<uint4*>(t + 2048 + o) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async();
  }
  const int32_t prev = __shfl_up_sync(0xffffffffu, id, 1);
  const uint32_t breaks = __ballot_sync(0xffffffffu, active && p > 0 && p < full && id != prev + 1);
  const bool one_run = ((breaks >> (lane & ~7)) & 0xffu) == 0;
  if (active && p == 0)
    mbar_expect_tx(bar, full * tile + (full < nvp && rows > 0 ? (base ? 2u : 1u) * rows * rb : 0u));
  __syncwarp();
  if (active) {
    if (one_run) {
      if (p == 0 && full > 0) bulk_g2s(dst, pool + (int64_t)id * tile, full * tile, bar);
    } else if (p < full) {
      bulk_g2s(dst + p * tile, pool + (int64_t)id * tile, tile, bar);
    }
    if (full < nvp && rows > 0 && p == full) {  // the lane holding the partial page
      const uint8_t* src = pool + (int64_t)id * tile;
      bulk_g2s(dst + full * tile, src, rows * rb, bar);
      if (base) bulk_g2s(dst + full * tile + 2048, src + 2048, rows * rb, bar);
    }
  }
}

// Reduce eight values per lane over the 32 lanes of a warp (max or sum), transposed so
// that nine shuffles suffice: lane l ends with the reduction of value l / 4.
template <bool kMax>
__device__ __forceinline__ float warp_reduce8(const float* v_in, int lane) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = v_in[i];
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // lanes with bit 4 set keep values 4..7
    const bool hi = lane & 16;
    const float keep = hi ? v[i + 4] : v[i], give = hi ? v[i] : v[i + 4];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, give, 16));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // bit 3: values 2..3 of the four left
    const bool hi = lane & 8;
    const float keep = hi ? v[i + 2] : v[i], give = hi ? v[i] : v[i + 2];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, give, 8));
  }
  {
    const bool hi = lane & 4;
    const float keep = hi ? v[1] : v[0], give = hi ? v[0] : v[1];
    v[0] = op(keep, __shfl_xor_sync(0xffffffffu, give, 4));
  }
  v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 2));
  v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
  return v[0];
}

// Reduce four values per lane over a warp (max or sum), transposed: six shuffles, and lane l
// ends with the reduction of value (l / 8) % 4.
template <bool kMax>
__device__ __forceinline__ float warp_reduce4(const float* v_in, int lane) {
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
  float v[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {  // lanes with bit 4 set keep values 2..3
    const bool hi = lane & 16;
    const float keep = hi ? v_in[i + 2] : v_in[i], give = hi ? v_in[i] : v_in[i + 2];
    v[i] = op(keep, __shfl_xor_sync(0xffffffffu, give, 16));
  }
  const bool hi = lane & 8;
  float r = op(hi ? v[1] : v[0], __shfl_xor_sync(0xffffffffu, hi ? v[0] : v[1], 8));
  r = op(r, __shfl_xor_sync(0xffffffffu, r, 4));
  r = op(r, __shfl_xor_sync(0xffffffffu, r, 2));
  r = op(r, __shfl_xor_sync(0xffffffffu, r, 1));
  return r;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// kG: query heads per KV head rounded up to 4 or 8 (the softmax works on kG score columns).
// The CTA works through its units back to back; every role counts blocks and steps over all
// of them (global counters), so the buffer rings and barrier phases simply continue from one
// unit into the next.
template <int kG>
__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // swizzled operand tiles need a 1024-byte aligned window
    if (threadIdx.x == 0) flag_status(a.status, kDevBadArg);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + 384);
  float* s_red = reinterpret_cast<float*>(smem + 512);      // [2][4 warps][8] block maxima
  float* s_mref = reinterpret_cast<float*>(smem + 768);     // [4 warps][4 agents][8] reference maxima
  int32_t* s_lp = reinterpret_cast<int32_t*>(smem + 1280);  // [4 warps][4 agents][2] length, position

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;
  int first, n_units;
  cta_units(a, first, n_units);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;  // a single arrival: the producer's expect_tx or one MMA commit
      if (i == kKEmpty0 || i == kKEmpty1 || i == kUFree || (i >= kKFFull0 && i <= kKFFull2))
        count = kRopeWarps;  // one arrival per RoPE warp
      if ((i >= kSFree0 && i <= kSFree2) || i == kPFull0 || i == kPFull1 || i == kRed0 || i == kRed1 ||
          i == kEpiDone)
        count = 4;  // one arrival per softmax warp
      mbar_init(&bars[i], count);
    }
    mbar_fence_init();
  }
  for (int i = threadIdx.x; i < 2 * kResSlotBytes / 16; i += kThreads) {  // the two constant ones tiles
    const int grp = i / (kResSlotBytes / 16), o = i % (kResSlotBytes / 16);
    *reinterpret_cast<uint4*>(smem + kOffVr + grp * kVrGroupBytes + 4 * kResSlotBytes + 16 * o) =
        make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  }
  if (threadIdx.x < 64) *reinterpret_cast<uint4*>(smem + kOffQZero + 16 * threadIdx.x) = make_uint4(0u, 0u, 0u, 0u);
  tc::fence_proxy_async();
  if (warp == 1) tc::alloc(s_tmem, kTmCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = *s_tmem;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    // Per block, in order: K tiles, each agent's k_res tiles, then V tiles and each agent's
    // v_res tiles (released together by the block's value products).  A block's page ids are
    // fetched one block ahead, one per lane: lane p < 8 the base page p, lane 8 a + p the
    // residual page p of agent a.  Every wait is for the buffer's previous user, two blocks
    // (or four k_res slots) back.
    int gb = 0, gn = 0;  // blocks and steps of every earlier unit
    int kb = 0, kn = 0, vb = 0;  // blocks / k_res steps / blocks of V whose copies went out
    bool ok = true;
    for (int k = 0; k < n_units && ok; ++k) {
      const Unit u = load_unit(a, first, k);
      const int na = u.na, nb = u.blocks();
      const uint8_t* kpool = a.k_base + (int64_t)u.h * a.num_base_pages * kBaseTile;
      const uint8_t* vpool = a.v_base + (int64_t)u.h * a.num_base_pages * kBaseTile;
      const int pg = lane & 7, ag = lane >> 3;
      const bool res_lane = ag < na;  // lanes of the agents' residual groups
      const int32_t my_agent = u.agent(res_lane ? ag : 0);
      const int32_t Lx = res_lane ? min(a.seq_lens[my_agent], a.max_seq_len) : 0;
      int32_t Lmax = Lx;  // rows at or past the longest sequence of the group are never read as data
#pragma unroll
      for (int o = 8; o < 32; o <<= 1) Lmax = max(Lmax, __shfl_xor_sync(0xffffffffu, Lmax, o));
      auto load_ids = [&](int b, int32_t& bid, int32_t& rid) {
        const int pbase = u.p0 + b * kBlockPages;
        const int nvp = min(kBlockPages, u.p1 - pbase);
        bid = rid = 0;
        if (lane < nvp) bid = a.bpt[(int64_t)u.agents[0] * a.pt_stride + pbase + lane];
        if (res_lane && pg < nvp) rid = a.rpt[(int64_t)my_agent * a.pt_stride + pbase + pg];
      };
      int32_t bid_next = 0, rid_next = 0;
      if (nb > 0) load_ids(0, bid_next, rid_next);
      for (int b = 0; b < nb; ++b) {
        const int g = gb + b;  // global block
        const int pbase = u.p0 + b * kBlockPages;
        const int nvp = min(kBlockPages, u.p1 - pbase);
        int32_t bid = bid_next, rid = rid_next;
        if (b + 1 < nb) load_ids(b + 1, bid_next, rid_next);
        if ((uint32_t)bid >= (uint32_t)a.num_base_pages) {
          flag_status(a.status, kDevBadPage);
          bid = 0;
        }
        if ((uint32_t)rid >= (uint32_t)a.num_res_pages) {
          flag_status(a.status, kDevBadPage);
          rid = 0;
        }
        // K tiles
        if (g >= 2 && !mbar_wait(&bars[kKEmpty0 + (g & 1)], ((g >> 1) - 1) & 1, a.status)) {
          ok = false;
          break;
        }
        copy_group(kpool, true, bid, nvp, kPage, smem + kOffK + (g & 1) * kBlockTiles, &bars[kKFull0 + (g & 1)],
                   lane < kBlockPages, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kKFull0 + (g & 1)]);
        kb = g + 1;
        // every agent's k_res tiles, one k_res slot (and barrier) per (block, agent) step
        for (int x = 0; x < na && ok; ++x) {
          const int n = gn + b * na + x;
          if (n >= kResSlots) ok = mbar_wait(&bars[kKrEmpty0 + (n & 3)], ((n >> 2) - 1) & 1, a.status);
        }
        if (!ok) break;
        const int kslot = (gn + b * na + ag) & 3;
        copy_group(a.k_res, false, rid, nvp, kPage, smem + kOffKr + kslot * kResSlotBytes, &bars[kKrFull0 + kslot],
                   res_lane, lane);
        __syncwarp();
        if (res_lane && pg == 0) mbar_arrive(&bars[kKrFull0 + kslot]);
        kn = gn + b * na + na;
        // V tiles and every agent's v_res tiles, on one barrier (released by the block's value products)
        if (g >= 2 && !mbar_wait(&bars[kVEmpty0 + (g & 1)], ((g >> 1) - 1) & 1, a.status)) {
          ok = false;
          break;
        }
        uint64_t* vbar = &bars[kVFull0 + (g & 1)];
        const int last = (pbase + nvp - 1) * kPage;  // first key of the block's last page
        copy_group(vpool, true, bid, nvp, min(kPage, max(0, Lmax - last)), smem + kOffV + (g & 1) * kBlockTiles, vbar,
                   lane < kBlockPages, lane);
        copy_group(a.v_res, false, rid, nvp, min(kPage, max(0, Lx - last)),
                   smem + kOffVr + (g & 1) * kVrGroupBytes + (4 - na + ag) * kResSlotBytes, vbar, res_lane, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(vbar);
        vb = g + 1;
      }
      gb += nb;
      gn += nb * na;
    }
    // never leave with copies in flight: the last phase of every barrier written to
    for (int b = max(0, kb - 2); b < kb; ++b) mbar_wait(&bars[kKFull0 + (b & 1)], (b >> 1) & 1, a.status);
    for (int b = max(0, vb - 2); b < vb; ++b) mbar_wait(&bars[kVFull0 + (b & 1)], (b >> 1) & 1, a.status);
    for (int n = max(0, kn - kResSlots); n < kn; ++n) mbar_wait(&bars[kKrFull0 + (n & 3)], (n >> 2) & 1, a.status);
  } else if (warp == 1) {
    // ------------------------------ U issuer ------------------------------
    //   U = Kr . B_k   [128 keys x 128]   per (block, agent).  Per unit the warp stages B_k of
    //   its head for every agent, as [16 ranks][128 d] in the base-tile layout (an MN-major
    //   operand), once the previous unit's products are done with the old one.
    const uint32_t idU = tc::idesc_bf16(128, 128, 0, 1);
    const uint32_t sBase = smem_u32(smem);
    const uint64_t dKr = tc::smem_desc(sBase + kOffKr, 16, 256, tc::kSwizzle32B);
    const uint64_t dBk = tc::smem_desc(sBase + kOffBk, 2048, 1024, tc::kSwizzle128B);
    int gn = 0;
    bool ok = true;
    for (int k = 0; k < n_units && ok; ++k) {
      const Unit u = load_unit(a, first, k);
      const int na = u.na, N = u.blocks() * na;
      if (k > 0) {  // every U of the previous unit is done with B_k
        if (lane == 0) {
          tc::commit(&bars[kUUnit]);
          ok = mbar_wait(&bars[kUUnit], (k - 1) & 1, a.status);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      for (int x = 0; x < na; ++x) {
        int32_t adapter = a.adapter_ids ? a.adapter_ids[u.agent(x)] : u.agent(x);
        if ((uint32_t)adapter >= (uint32_t)a.n_adapters) {
          flag_status(a.status, kDevBadArg);
          adapter = 0;
        }
        const __nv_bfloat16* B = a.B_k + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)u.h * kHeadDim;
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // 16 ranks x 16 chunks of 8 d
          const int c = lane + 32 * i, r = c >> 4, ch = c & 15;
          *reinterpret_cast<uint4*>(smem + kOffBk + x * 4096 + base_off(r, ch * 8)) =
              *reinterpret_cast<const uint4*>(B + (int64_t)r * a.hkv * kHeadDim + ch * 8);
        }
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        for (int n = 0; n < N && ok; ++n) {
          const int m = gn + n;
          ok = mbar_wait(&bars[kKrFull0 + (m & 3)], (m >> 2) & 1, a.status) &&
               (m < 1 || mbar_wait(&bars[kUFree], (m - 1) & 1, a.status));
          if (!ok) break;
          tc::fence_after();
          tc::mma_ss(tm + kTmU, dKr + (m & 3) * (kResSlotBytes >> 4), dBk + (n % na) * (4096 >> 4), idU, 0);
          tc::commit(&bars[kUFull]);
          tc::commit(&bars[kKrEmpty0 + (m & 3)]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      gn += N;
    }
    if (lane == 0) {
      tc::commit(&bars[kMmaDone]);  // never leave with MMAs in flight
      mbar_wait(&bars[kMmaDone], 0, a.status);
    }
    __syncwarp();
  } else if (warp == kScoreWarp) {
    // ------------------------------ score issuer ------------------------------
    //   S = K . Q^T      [128 keys x 16]    K from tensor memory, per (block, agent).  Per unit the
    //   warp stages Q^T of every agent: [2 halves][8 rows (query heads, zero past G)][128 B]; the
    //   second 8-row group (query heads 8..15) reads a shared block of zeros.
    const uint32_t idS = tc::idesc_bf16(128, 16, 0, 0);
    const uint32_t sBase = smem_u32(smem);
    int gn = 0;
    bool ok = true;
    for (int k = 0; k < n_units && ok; ++k) {
      const Unit u = load_unit(a, first, k);
      const int na = u.na, N = u.blocks() * na;
      if (k > 0) {  // every S of the previous unit is done with Q^T
        if (lane == 0) {
          tc::commit(&bars[kSUnit]);
          ok = mbar_wait(&bars[kSUnit], (k - 1) & 1, a.status);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      for (int x = 0; x < na; ++x) {
        const int32_t agent = u.agent(x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // 8 query-head rows x 16 chunks of 8 d
          const int c = lane + 32 * i, g = c >> 4, ch = c & 15;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (g < G)
            v = *reinterpret_cast<const uint4*>(a.q + ((int64_t)agent * a.hkv * G + (int64_t)u.h * G + g) * kHeadDim + ch * 8);
          *reinterpret_cast<uint4*>(smem + kOffQ + x * 2048 + tc::sw128_off(8, g, ch * 8)) = v;
        }
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        for (int n = 0; n < N && ok; ++n) {
          const int m = gn + n;
          const int sr = m % kRing, sp = (m / kRing) & 1;  // ring slot and phase parity of step m
          ok = mbar_wait(&bars[kKFFull0 + sr], sp, a.status) &&
               (m < kRing || mbar_wait(&bars[kSFree0 + sr], sp ^ 1, a.status));
          if (!ok) break;
          tc::fence_after();
          const uint32_t q = kOffQ + (n % na) * 2048;  // the two 64-column halves of Q^T at q, q + 1024
          const uint64_t dq0 = tc::smem_desc(sBase + q, 16, kOffQZero - q, tc::kSwizzle128B);
          const uint64_t dq1 = tc::smem_desc(sBase + q + 1024, 16, kOffQZero - q - 1024, tc::kSwizzle128B);
          const uint32_t dS = tm + kTmS + 16 * sr, aK = tm + kTmKF + 64 * sr;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // K = 16 per step: 8 TMEM columns of A, 32 bytes of B
            tc::mma_ts(dS, aK + 8 * ks, (ks < 4 ? dq0 : dq1) + 2 * (ks & 3), idS, ks > 0);
          tc::commit(&bars[kSFull0 + sr]);
          tc::commit(&bars[kKFFree0 + sr]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      gn += N;
    }
    if (lane == 0) {
      tc::commit(&bars[kSDone]);
      mbar_wait(&bars[kSDone], 0, a.status);
    }
    __syncwarp();
  } else if (warp < kSoftWarp0) {
    // ------------------------------ RoPE group ------------------------------
    // Two warps per TMEM lane quadrant; warp half hf owns K columns [32 hf, 32 hf + 32)
    // and [64 + 32 hf, 96 + 32 hf) of its 32 keys.
    const int q4 = warp & 3, hf = (warp - 2) >> 2;
    const int row = 32 * q4 + lane;  // key row of the block == TMEM lane
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);
    const int pg = row >> 4, t = row & 15;
    int gb = 0, gn = 0;
    bool ok = true;
    uint4 rp[2][4];  // rotation groups of this warp's two column chunks for key j (see below)
    for (int k = 0; k < n_units && ok; ++k) {
      const Unit u = load_unit(a, first, k);
      const int na = u.na, N = u.blocks() * na;
      for (int n = 0; n < N && ok; ++n) {
        const int b = n / na, ai = n - b * na;
        const int g = gb + b, m = gn + n;  // global block and step
        const int stage = g & 1;
        const int pbase = u.p0 + b * kBlockPages;
        const int j = pbase * kPage + row;
        if (ai == 0) {
          // chunk c = 32 hf + 16 cc holds frequency groups m = c/2 .. c/2 + 7: 32-byte units
          // c/8 and c/8 + 1 of the row, stored at unit u ^ (j % 8)
          const int jr = j < a.rope_positions ? j : 0;
          const uint4* rrow = reinterpret_cast<const uint4*>(a.rope + (int64_t)jr * kRopeRow);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
              const int un = 4 * hf + 2 * cc + uu;
              rp[cc][2 * uu] = __ldg(rrow + (un ^ (j & 7)) * 2);
              rp[cc][2 * uu + 1] = __ldg(rrow + (un ^ (j & 7)) * 2 + 1);
            }
          ok = mbar_wait(&bars[kKFull0 + stage], (g >> 1) & 1, a.status);
          if (!ok) break;
        }
        // U of this step, read out at once (as bf16 pairs) so that the next U can go ahead
        ok = mbar_wait(&bars[kUFull], m & 1, a.status);
        if (!ok) break;
        tc::fence_after();
        uint32_t ul[2][8], uh[2][8];  // [chunk][pair]: U columns (c + 2 i, c + 2 i + 1) and + 64
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 32 * hf + 16 * cc;
          uint32_t lo[16], hi[16];
          tc::ld16(tl + kTmU + c, lo);
          tc::ld16(tl + kTmU + 64 + c, hi);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ul[cc][i] = pack_bf16(__uint_as_float(lo[2 * i]), __uint_as_float(lo[2 * i + 1]));
            uh[cc][i] = pack_bf16(__uint_as_float(hi[2 * i]), __uint_as_float(hi[2 * i + 1]));
          }
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kUFree]);
        const int kr = m % kRing, kp = (m / kRing) & 1;
        if (m >= kRing && !mbar_wait(&bars[kKFFree0 + kr], kp ^ 1, a.status)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint8_t* kt = smem + kOffK + stage * kBlockTiles + pg * kBaseTile;
        const uint32_t kf = tl + kTmKF + 64 * kr;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {  // d in [c, c + 16) and [c + 64, c + 80)
          const int c = 32 * hf + 16 * cc;
          uint4 kl[2], kh[2];
          kl[0] = *reinterpret_cast<const uint4*>(kt + base_off(t, c));
          kl[1] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 8));
          kh[0] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 64));
          kh[1] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 72));
          const uint32_t* klw = reinterpret_cast<const uint32_t*>(kl);
          const uint32_t* khw = reinterpret_cast<const uint32_t*>(kh);
          uint32_t olo[8], ohi[8];
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) {  // frequency group c/2 + i2: frequencies of d = c + 2 i2, + 1
            const uint4 w = rp[cc][(i2 >> 2) * 2 + ((i2 & 3) >> 1)];
            const uint32_t cw = (i2 & 1) ? w.z : w.x, sw = (i2 & 1) ? w.w : w.y;
            // the rotated residual term in bf16x2 (its roundings are at the residual's scale), then
            // one bf16 rounding of K = Kb + RoPE_j(U)
            const __nv_bfloat162 C = *reinterpret_cast<const __nv_bfloat162*>(&cw);
            const __nv_bfloat162 S = *reinterpret_cast<const __nv_bfloat162*>(&sw);
            const __nv_bfloat162 UL = *reinterpret_cast<const __nv_bfloat162*>(&ul[cc][i2]);
            const __nv_bfloat162 UH = *reinterpret_cast<const __nv_bfloat162*>(&uh[cc][i2]);
            const __nv_bfloat162 rl = __hfma2(__hneg2(UH), S, __hmul2(UL, C));
            const __nv_bfloat162 rh = __hfma2(UH, C, __hmul2(UL, S));
            const __nv_bfloat162 kl2 = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&klw[i2]), rl);
            const __nv_bfloat162 kh2 = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&khw[i2]), rh);
            olo[i2] = *reinterpret_cast<const uint32_t*>(&kl2);
            ohi[i2] = *reinterpret_cast<const uint32_t*>(&kh2);
          }
          tc::st8(kf + (c >> 1), olo);       // K columns d < 64: bf16 pairs (d, d + 1) at column d / 2
          tc::st8(kf + 32 + (c >> 1), ohi);  // K columns d >= 64
        }
        tc::wait_st();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kKFFull0 + kr]);
          if (ai == na - 1) mbar_arrive(&bars[kKEmpty0 + stage]);
        }
      }
      gb += u.blocks();
      gn += N;
    }
  } else if (warp == kValueWarp) {
    // ------------------------------ value products ------------------------------
    // Per block, for all its agents at once (B = P^T of every agent side by side,
    // 8 columns each):
    //   O^T += Vb^T . P^T                  [128 d x 8 na]
    //   R   += [Vr^T of each agent; 1] . P^T  [128 x 8 na]
    // The second product's A operand stacks 16-row atoms 4 KB apart: Vr^T of agents
    // 0..na-1 (rows 16 a .. 16 a + 15), then a tile of ones (rows 16 na ..).  Rows
    // 16 a + r, columns 8 a + g of R hold acc_r^T[r][g] of agent a, and rows 16 na ..
    // hold l[g] = sum over keys of P for every agent; the other cells are cross terms,
    // never read.  A unit's first block overwrites O and R once the epilogue of the
    // previous unit has read them.
    if (lane == 0) {
      const uint32_t sBase = smem_u32(smem);
      const uint64_t dV = tc::smem_desc(sBase + kOffV, 2048, 1024, tc::kSwizzle128B);
      const uint64_t dP = tc::smem_desc(sBase + kOffP, 4096, 256, tc::kSwizzle32B);
      int gb = 0;
      bool ok = true;
      for (int k = 0; k < n_units && ok; ++k) {
        const Unit u = load_unit(a, first, k);
        const int na = u.na, nb = u.blocks();
        const uint32_t idV = tc::idesc_bf16(128, na > 2 ? 32 : 16, 1, 1);
        const uint64_t dR =
            tc::smem_desc(sBase + kOffVr + (4 - na) * kResSlotBytes, kResSlotBytes, 256, tc::kSwizzle32B);
        if (k > 0) ok = mbar_wait(&bars[kEpiDone], (k - 1) & 1, a.status);
        for (int b = 0; b < nb && ok; ++b) {
          const int g = gb + b;
          ok = mbar_wait(&bars[kVFull0 + (g & 1)], (g >> 1) & 1, a.status) &&
               mbar_wait(&bars[kPFull0 + (g & 1)], (g >> 1) & 1, a.status);
          if (!ok) break;
          tc::fence_after();
          const int nvp = min(kBlockPages, u.p1 - (u.p0 + b * kBlockPages));
          const uint64_t dv = dV + (g & 1) * (kBlockTiles >> 4), dp = dP + (g & 1) * (8192 >> 4);
          const uint64_t dr = dR + (g & 1) * (kVrGroupBytes >> 4);  // 8 atoms of 16 rows, 4 KB apart
          const uint32_t acc0 = b > 0;
#pragma unroll
          for (int ks = 0; ks < kBlockPages; ++ks)  // one page (16 keys) per step
            if (ks < nvp) tc::mma_ss(tm + kTmO, dv + ks * (kBaseTile >> 4), dp + ks * (512 >> 4), idV, acc0 | (ks > 0));
#pragma unroll
          for (int ks = 0; ks < kBlockPages; ++ks)
            if (ks < nvp) tc::mma_ss(tm + kTmR, dr + ks * (kResTile >> 4), dp + ks * (512 >> 4), idV, acc0 | (ks > 0));
          tc::commit(&bars[kPFree0 + (g & 1)]);
          tc::commit(&bars[kODone0 + (g & 1)]);
          tc::commit(&bars[kVEmpty0 + (g & 1)]);
        }
        gb += nb;
      }
      tc::commit(&bars[kValDone]);
      mbar_wait(&bars[kValDone], 0, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax group ------------------------------
    const int sw_ = warp & 3;
    const int row = 32 * sw_ + lane;  // key row of the block == TMEM lane (and d row of O^T)
    const uint32_t tl = tm + ((uint32_t)(32 * sw_) << 16);
    float* mref = s_mref + sw_ * (kMaxGroup * 8);  // this warp's copy (all four evolve identically)
    int32_t* lp = s_lp + sw_ * (kMaxGroup * 2);    // this warp's copy of each agent's (length, position)
    // query head whose warp-wide reductions this lane ends up holding, and the lanes that publish them
    const int gl = kG == 8 ? lane >> 2 : lane >> 3;
    const bool publisher = kG == 8 ? (lane & 3) == 0 : (lane & 7) == 0;
    int gb = 0, gn = 0;
    bool ok = true;
    for (int k = 0; k < n_units && ok; ++k) {
      const Unit u = load_unit(a, first, k);
      const int na = u.na, nb = u.blocks(), N = nb * na;
      __syncwarp();
      mref[lane] = -INFINITY;  // 4 agents x 8 query heads
      if (lane < kMaxGroup) {
        const int32_t agent = u.agent(lane);
        const int32_t L = a.seq_lens[agent], pos = a.positions[agent];
        lp[2 * lane] = lane < na ? min(L, a.max_seq_len) : 0;
        lp[2 * lane + 1] = pos;
        if (lane < na && sw_ == 0 && u.h == 0 && (L < 1 || L > a.max_seq_len || pos < 0 || pos >= L))
          flag_status(a.status, kDevBadArg);
      }
      __syncwarp();
      for (int n = 0; n < N && ok; ++n) {
        const int b = n / na, ai = n - b * na;
        const int g = gb + b, m = gn + n;  // global block and step
        const int pbase = u.p0 + b * kBlockPages;
        const int j = pbase * kPage + row;
        const int32_t L = lp[2 * ai], pos = lp[2 * ai + 1];
        const bool vis = j < L && j <= pos && j < u.p1 * kPage;
        const int sr = m % kRing;
        ok = mbar_wait(&bars[kSFull0 + sr], (m / kRing) & 1, a.status);
        if (!ok) break;
        tc::fence_after();
        uint32_t sv[kG];
        if constexpr (kG == 8) tc::ld8(tl + kTmS + 16 * sr, sv);
        else tc::ld4(tl + kTmS + 16 * sr, sv);
        tc::wait_ld();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSFree0 + sr]);
        float sc[kG];
#pragma unroll
        for (int q = 0; q < kG; ++q) sc[q] = (vis && q < G) ? __uint_as_float(sv[q]) * a.scale_log2 : -INFINITY;
        float wmax;  // max over the warp's keys of query head gl
        if constexpr (kG == 8) wmax = warp_reduce8<true>(sc, lane);
        else wmax = warp_reduce4<true>(sc, lane);
        float* red = s_red + (m & 1) * 32;
        if (publisher) red[sw_ * kG + gl] = wmax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kRed0 + (m & 1)]);
        // while the other warps' maxima come in: probabilities against the current reference
        float mr[kG], ps[kG];
#pragma unroll
        for (int q = 0; q < kG; ++q) {
          mr[q] = mref[ai * 8 + q];
          ps[q] = (vis && q < G) ? ex2(sc[q] - (mr[q] == -INFINITY ? 0.f : mr[q])) : 0.f;
        }
        ok = mbar_wait(&bars[kRed0 + (m & 1)], (m >> 1) & 1, a.status);
        if (!ok) break;
        // lazy rescale: keep the reference maximum unless the block maximum passes it by 2^8
        float alpha[kG];
        bool need_any = false;
#pragma unroll
        for (int q = 0; q < kG; ++q) {
          const float bm = fmaxf(fmaxf(red[q], red[kG + q]), fmaxf(red[2 * kG + q], red[3 * kG + q]));
          const bool need = q < G && bm > mr[q] + 8.f;
          need_any |= need;
          alpha[q] = (need && mr[q] != -INFINITY) ? ex2(mr[q] - bm) : 1.f;
          if (need) mr[q] = bm;
        }
        if (need_any) {  // uniform across the group: every warp saw the same maxima
          float ml = mr[0];
#pragma unroll
          for (int q = 1; q < kG; ++q)
            if (gl == q) ml = mr[q];
          __syncwarp();
          if (publisher) mref[ai * 8 + gl] = ml;
#pragma unroll
          for (int q = 0; q < kG; ++q) ps[q] = (vis && q < G) ? ex2(sc[q] - mr[q]) : 0.f;
          if (b > 0) {
            // O^T and R are stable once the value products of block g - 1 are done (one barrier
            // per block parity, so a wait is never more than one phase ahead of the barrier)
            ok = mbar_wait(&bars[kODone0 + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status);
            if (!ok) break;
            tc::fence_after();
            uint32_t ov[kG], rv[kG];
            if constexpr (kG == 8) {
              tc::ld8(tl + kTmO + 8 * ai, ov);
              tc::ld8(tl + kTmR + 8 * ai, rv);
            } else {
              tc::ld4(tl + kTmO + 8 * ai, ov);
              tc::ld4(tl + kTmR + 8 * ai, rv);
            }
            tc::wait_ld();
#pragma unroll
            for (int q = 0; q < kG; ++q) {
              ov[q] = __float_as_uint(__uint_as_float(ov[q]) * alpha[q]);
              rv[q] = __float_as_uint(__uint_as_float(rv[q]) * alpha[q]);
            }
            if constexpr (kG == 8) {
              tc::st8(tl + kTmO + 8 * ai, ov);
              tc::st8(tl + kTmR + 8 * ai, rv);
            } else {
              tc::st4(tl + kTmO + 8 * ai, ov);
              tc::st4(tl + kTmR + 8 * ai, rv);
            }
            tc::wait_st();
            tc::fence_before();
          }
        }
        uint32_t pw[4] = {0u, 0u, 0u, 0u};  // P^T[key][g] in bf16, zero past G or for masked keys
#pragma unroll
        for (int q2 = 0; q2 < kG / 2; ++q2) pw[q2] = pack_bf16(ps[2 * q2], ps[2 * q2 + 1]);
        if (ai == 0 && g >= 2) ok = mbar_wait(&bars[kPFree0 + (g & 1)], ((g >> 1) - 1) & 1, a.status);
        if (!ok) break;
        // P^T of agent ai: columns 8 ai .. 8 ai + 7 = atom ai / 2, 16-byte chunk ai % 2 of each row
        uint8_t* pbuf = smem + kOffP + (g & 1) * 8192 + (ai >> 1) * 4096;
        *reinterpret_cast<uint4*>(pbuf + tc::sw32_off(row, (ai & 1) * 8)) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
        if (ai == na - 1) {
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kPFull0 + (g & 1)]);
        }
      }
      if (!ok) break;
      // epilogue: one partial (m, l, acc, acc_r) per (agent, head) of the unit
      const int glast = gb + nb - 1;
      if (nb > 0) ok = mbar_wait(&bars[kODone0 + (glast & 1)], (glast >> 1) & 1, a.status);
      tc::fence_after();
      if (u.slot_base >= 0) {
        for (int ai = 0; ai < na; ++ai) {
          uint32_t ov[8], rv[8];
          tc::ld8(tl + kTmO + 8 * ai, ov);
          tc::ld8(tl + kTmR + 8 * ai, rv);
          tc::wait_ld();
          const int64_t rec0 = ((int64_t)(u.slot_base + ai) * a.hkv + u.h) * G;
          const int r = row - kRank * ai;  // rank held by this lane of agent ai's rows of R
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < G) {
              a.part[(rec0 + q) * kPartCols + row] = nb > 0 ? __uint_as_float(ov[q]) : 0.f;
              if (r >= 0 && r < kRank) a.part[(rec0 + q) * kPartCols + kHeadDim + r] = nb > 0 ? __uint_as_float(rv[q]) : 0.f;
              if (row == kRank * na) {  // first row of the ones product: l
                a.ml[(rec0 + q) * 2] = nb > 0 ? mref[ai * 8 + q] : -INFINITY;
                a.ml[(rec0 + q) * 2 + 1] = nb > 0 ? __uint_as_float(rv[q]) : 0.f;
              }
            }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kEpiDone]);  // O and R may be overwritten now
      gb += nb;
      gn += N;
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tm, kTmCols);
  }
}

struct CombineArgs {
  const float* part;
  const float* ml;
  const int32_t* csr_off;    // plan mode: [A+1]
  const int32_t* csr_slots;  // plan mode: slot ids
  int32_t chunks;            // no-plan mode: slots of agent a are [a*chunks, (a+1)*chunks)
  int32_t n_slots;
  uint32_t* status;
  int32_t hkv, G;
  const __nv_bfloat16* B_v;
  const int32_t* adapter_ids;
  int32_t n_adapters;
  __nv_bfloat16* out;        // [A][Hq][128]
};

constexpr int kCombineSlots = 1024;  // slots handled per pass

// One CTA per (agent, KV head, query head): log-sum-exp merge of the agent's
// partials, then out = (acc + acc_r B_v[:, hD:(h+1)D]) / l.  All partial loads
// of a pass are independent, so their latencies overlap.
__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ CombineArgs a) {
  const int agent = blockIdx.x, h = blockIdx.y, gq = blockIdx.z, d = threadIdx.x;
  const int G = a.G;
  __shared__ float s_w[kCombineSlots];
  __shared__ int32_t s_slot[kCombineSlots];
  __shared__ float s_red[4];
  __shared__ float s_accr[kRank];
  int32_t s_begin, s_end;
  if (a.csr_off) {
    s_begin = a.csr_off[agent];
    s_end = a.csr_off[agent + 1];
  } else {
    s_begin = agent * a.chunks;
    s_end = s_begin + a.chunks;
  }
  if (s_begin < 0 || s_end < s_begin || s_end > a.n_slots) {
    if (d == 0) flag_status(a.status, kDevBadArg);
    s_end = s_begin = 0;
  }
  int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
  if ((uint32_t)adapter >= (uint32_t)a.n_adapters) adapter = 0;
  const __nv_bfloat16* Bv = a.B_v + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim + d;
  float bv[kRank];
#pragma unroll
  for (int k = 0; k < kRank; ++k) bv[k] = __bfloat162float(Bv[(int64_t)k * a.hkv * kHeadDim]);

  // pass 1: global maximum of the reference maxima
  float M = -INFINITY;
  for (int i = s_begin + d; i < s_end; i += 128) {
    int32_t slot = a.csr_off ? a.csr_slots[i] : i;
    if ((uint32_t)slot >= (uint32_t)a.n_slots) slot = -1;
    if (slot >= 0) M = fmaxf(M, a.ml[(((int64_t)slot * a.hkv + h) * G + gq) * 2]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if ((d & 31) == 0) s_red[d >> 5] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));

  float acc = 0.f, accr = 0.f, lsum = 0.f;
  for (int b0 = s_begin; b0 < s_end; b0 += kCombineSlots) {
    const int nb = min(kCombineSlots, s_end - b0);
    __syncthreads();
    for (int i = d; i < nb; i += 128) {
      int32_t slot = a.csr_off ? a.csr_slots[b0 + i] : b0 + i;
      float w = 0.f;
      if ((uint32_t)slot < (uint32_t)a.n_slots) {
        const float m = a.ml[(((int64_t)slot * a.hkv + h) * G + gq) * 2];
        w = (m == -INFINITY || M == -INFINITY) ? 0.f : exp2f(m - M);
      } else {
        slot = 0;
      }
      s_w[i] = w;
      s_slot[i] = slot;
    }
    __syncthreads();
#pragma unroll 8
    for (int i = 0; i < nb; ++i) {
      const float w = s_w[i];
      const int64_t rec = ((int64_t)s_slot[i] * a.hkv + h) * G + gq;
      acc += w * a.part[rec * kPartCols + d];
      if (d < kRank) accr += w * a.part[rec * kPartCols + kHeadDim + d];
      if (d == 0) lsum += w * a.ml[rec * 2 + 1];
    }
  }
  if (d < kRank) s_accr[d] = accr;
  if (d == 0) s_red[0] = lsum;
  __syncthreads();
  float o = acc;
#pragma unroll
  for (int k = 0; k < kRank; ++k) o += s_accr[k] * bv[k];
  lsum = s_red[0];
  o = lsum > 0.f ? o / lsum : 0.f;
  a.out[((int64_t)agent * a.hkv * G + (int64_t)h * G + gq) * kHeadDim + d] = __float2bfloat16_rn(o);
}

}  // namespace

DecodeGeometry decode_geometry(const forkkv_attn_params& p) {
  DecodeGeometry g{};
  const int32_t G = p.num_q_heads / p.num_kv_heads;
  if (p.plan) {
    g.n_items = p.plan_items;
    g.n_slots = p.plan_slots;
  } else {
    // Split every agent's pages into `chunks` items of `chunk_pages` pages (a multiple of
    // the 8 pages of a block) so that the A * chunks * Hkv units fill the SMs without
    // passing one unit per SM (a second, partial round would double the time).
    const int32_t max_pages = (p.max_seq_len + kPage - 1) / kPage;
    const int64_t want = 152;  // one CTA per SM
    int32_t chunks = (int32_t)(want / ((int64_t)p.n_agents * p.num_kv_heads));
    chunks = max(1, min(chunks, (max_pages + 7) / 8));
    int32_t chunk_pages = (max_pages + chunks - 1) / chunks;
    chunk_pages = max(kBlockPages, (chunk_pages + kBlockPages - 1) / kBlockPages * kBlockPages);
    chunks = (max_pages + chunk_pages - 1) / chunk_pages;
    g.chunks = max(1, chunks);
    g.chunk_pages = chunk_pages;
    g.n_items = p.n_agents * g.chunks;
    g.n_slots = g.n_items;
  }
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  g.partial_bytes = up((size_t)g.n_slots * p.num_kv_heads * G * kPartCols * sizeof(float));
  g.ml_bytes = up((size_t)g.n_slots * p.num_kv_heads * G * 2 * sizeof(float));
  g.rope_bytes = p.rope_table ? 0 : up((size_t)((p.max_seq_len + kPage - 1) / kPage * kPage) * kRopeRow);
  g.total_bytes = g.partial_bytes + g.ml_bytes + g.rope_bytes;
  return g;
}

cudaError_t launch_decode(const forkkv_attn_params& p, const DecodeGeometry& g, const void* rope_table,
                          uint32_t* status, cudaStream_t stream) {
  static thread_local int configured_device = -1, sm_count = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_split_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_split_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int32_t G = p.num_q_heads / p.num_kv_heads;
  const int64_t base_layer = (int64_t)p.pools.num_base_pages * p.pools.num_kv_heads * kBaseTile;
  const int64_t res_layer = (int64_t)p.pools.num_res_pages * kResTile;
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);

  DecodeArgs a;
  a.k_base = static_cast<const uint8_t*>(p.pools.k_base) + p.layer * base_layer;
  a.v_base = static_cast<const uint8_t*>(p.pools.v_base) + p.layer * base_layer;
  a.k_res = static_cast<const uint8_t*>(p.pools.k_res) + p.layer * res_layer;
  a.v_res = static_cast<const uint8_t*>(p.pools.v_res) + p.layer * res_layer;
  a.num_base_pages = p.pools.num_base_pages;
  a.num_res_pages = p.pools.num_res_pages;
  a.hkv = p.num_kv_heads;
  a.G = G;
  a.q = static_cast<const __nv_bfloat16*>(p.q);
  a.bpt = p.bpt;
  a.rpt = p.rpt;
  a.pt_stride = p.pt_stride;
  a.seq_lens = p.seq_lens;
  a.positions = p.positions;
  a.B_k = static_cast<const __nv_bfloat16*>(p.B_k);
  a.adapter_ids = p.adapter_ids;
  a.n_adapters = p.n_adapters;
  a.rope = static_cast<const uint8_t*>(rope_table);
  a.rope_positions = p.rope_table ? p.rope_table_positions : (p.max_seq_len + kPage - 1) / kPage * kPage;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.0f / sqrtf((float)kHeadDim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.plan = p.plan;
  a.n_items = g.n_items;
  if (p.plan) {  // the schedule follows the items and the per-agent slot lists
    a.cta_off = p.plan + (int64_t)p.plan_items * FORKKV_PLAN_ITEM_INTS + p.n_agents + 1 + p.plan_slots;
    a.units = a.cta_off + p.plan_ctas + 1;
    a.n_ctas = p.plan_ctas;
  } else {  // every (item, head) pair, dealt round-robin over at most one CTA per SM
    a.cta_off = a.units = nullptr;
    a.n_ctas = (int32_t)std::min<int64_t>((int64_t)g.n_items * p.num_kv_heads, std::max(1, sm_count));
  }
  a.chunk_pages = g.chunk_pages;
  a.chunks = g.chunks;
  a.n_agents = p.n_agents;
  a.max_seq_len = p.max_seq_len;
  a.n_slots = g.n_slots;
  a.part = reinterpret_cast<float*>(ws);
  a.ml = reinterpret_cast<float*>(ws + g.partial_bytes);
  a.status = status;
  if (G <= 4)
    decode_split_kernel<4><<<a.n_ctas, kThreads, kSmemBytes, stream>>>(a);
  else
    decode_split_kernel<8><<<a.n_ctas, kThreads, kSmemBytes, stream>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CombineArgs c;
  c.part = a.part;
  c.ml = a.ml;
  c.csr_off = p.plan ? p.plan + (int64_t)p.plan_items * FORKKV_PLAN_ITEM_INTS : nullptr;
  c.csr_slots = p.plan ? c.csr_off + p.n_agents + 1 : nullptr;
  c.chunks = g.chunks;
  c.n_slots = g.n_slots;
  c.status = status;
  c.hkv = p.num_kv_heads;
  c.G = G;
  c.B_v = static_cast<const __nv_bfloat16*>(p.B_v);
  c.adapter_ids = p.adapter_ids;
  c.n_adapters = p.n_adapters;
  c.out = static_cast<__nv_bfloat16*>(p.out);
  decode_combine_kernel<<<dim3(p.n_agents, p.num_kv_heads, G), 128, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace fkv
