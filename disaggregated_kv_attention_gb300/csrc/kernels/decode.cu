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
//     warp 1      allocates tensor memory; stages B_k of the unit's head and
//                 issues, per (block, agent):
//                   U    = Kr . B_k                 [128 keys x 128]  smem x smem
//     warp 15     stages Q of the unit's agents and issues, per (block, agent):
//                   S    = K . Q^T                  [128 keys x 16]   K from TMEM
//                 (K and S in rings of three in tensor memory)
//     warps 2..9  RoPE group, one key per thread and half of the columns per
//                 warp: K = Kb + RoPE_j(U) in bf16x2 fused multiply-adds onto Kb
//                 (K rounded twice at its own scale), written to tensor memory
//                 as the A operand of the score product
//     warps 10..13 softmax group, one key per thread: scores, length mask, block
//                 maxima across the group, lazy rescale of O (only when the
//                 running maximum grows by 2^8), P^T to shared memory; at the end
//                 of a unit one partial (m, l, acc, acc_r) per (agent, KV head)
//     warp 14     issues, per block and for all its agents at once,
//                   O^T += Vb^T . P^T  and  R += Vr^T . P^T (rank-16 value path)
//                 and l as the product of a tile of ones with P^T.
//   combine       one CTA per (agent, KV head, query head): log-sum-exp merge of
//                 the partials, then out = (acc + acc_r . B_v[:, hD:(h+1)D]) / l,
//                 B_v applied once per query head.
// The three issuer warps run their loops with all 32 lanes (descriptors and ring
// indices computed warp-uniformly) and issue each MMA and commit from one lane
// chosen by elect.sync.  Every wait is on an mbarrier with a bounded spin; a
// timeout sets the device status word instead of hanging.
#include <math.h>

#include <algorithm>

#include "../internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fkv {
namespace {

constexpr int kMaxGroup = 4;                 // agents per work unit
constexpr int kMaxGroupQ = 8;                // query heads per KV head
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

// tensor memory columns: U (fp32) in two buffers, so that the next step's U is computed
// while the rotation warps read this one; K (bf16 pairs) in a ring of 2 and S in a ring of
// 3; O^T [128 d x 8 agents' query heads] and the residual-value product
constexpr int kKfRing = 2, kSRing = 3;
constexpr uint32_t kTmU = 0, kTmKF = 256, kTmS = kTmKF + 64 * kKfRing, kTmO = 448, kTmR = 480, kTmCols = 512;
static_assert(kTmS + 16 * kSRing <= kTmO && kTmR + 32 <= kTmCols, "tensor memory regions overlap");

enum {
  kKFull0, kKFull1, kVFull0, kVFull1, kKEmpty0, kKEmpty1, kVEmpty0, kVEmpty1,
  kKrFull0, kKrFull1, kKrFull2, kKrFull3, kKrEmpty0, kKrEmpty1, kKrEmpty2, kKrEmpty3,
  kUFull0, kUFull1, kUFree0, kUFree1, kKFFull0, kKFFull1, kKFFree0, kKFFree1, kSFull0, kSFull1, kSFull2,
  kSFree0, kSFree1, kSFree2,
  kPFull0, kPFull1, kPFree0, kPFree1, kRed0, kRed1, kODone0, kODone1, kUUnit, kSUnit, kEpiDone, kUnitReady0, kUnitReady1, kUnitFree0, kUnitFree1,
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
  const int32_t* holes;  // [n_agents][2] slot map (first hole slot, hole length), or null
  const __nv_bfloat16* B_k;  // [n_adapters][16][Hkv*128]
  const int32_t* adapter_ids;
  int32_t n_adapters;
  const uint8_t* rope;
  int32_t rope_positions;
  float scale_log2;
  const int32_t* units;  // plan's unit records (FORKKV_PLAN_UNIT_INTS each), or null: units by formula
  int32_t n_units;       // plan: records; no plan: n_items * hkv
  int32_t chunk_pages, chunks;
  int32_t n_agents, max_seq_len, n_slots;
  float* part;
  float* ml;
  uint32_t* status;
};

// A unit of work is an item (a page range walked by a group of agents) for one KV head.  The
// producer warp describes each unit of its CTA, in order, in a ring of two descriptors in
// shared memory (kUnitInts int32 each, one field per lane when built) that the other warps
// read at the start of the unit.
constexpr int kUnitInts = 26;
enum {
  kUfP0, kUfP1, kUfNa, kUfH, kUfSlot, kUfEnd,  // page range, agents, KV head, first slot, end of list
  kUfAgent = 6, kUfL = 10, kUfPos = 14, kUfAdapter = 18,  // per agent (4 each): index, keys, position, adapter,
  kUfHole = 22                                           // hole (16 * first slot + length, 0: none)
};
constexpr int kOffUnits = 1408;  // 2 x kUnitInts int32 in the header of shared memory
constexpr int kOffHoles = 1664;  // the softmax warps' copies of each agent's hole end
static_assert(kOffUnits + 2 * kUnitInts * 4 <= kOffHoles && kOffHoles + 4 * kMaxGroup * 4 <= 2048,
              "unit ring and hole codes overlap each other or the operand tiles");

// The first unit of this CTA: plan record blockIdx.x, or unit code blockIdx.x (-1: none).
__device__ __forceinline__ int32_t first_unit(const DecodeArgs& a) {
  return (int32_t)blockIdx.x < a.n_units ? (int32_t)blockIdx.x : -1;
}

// Raw material of unit r, one int per lane: the plan record's words, or without a plan the
// unit agent's sequence length (lane 0), from which its chunk bounds follow.
__device__ __forceinline__ int32_t unit_raw(const DecodeArgs& a, int32_t r, int lane) {
  if (r < 0) return 0;
  if (a.units) return lane < FORKKV_PLAN_UNIT_INTS ? __ldg(a.units + (int64_t)r * FORKKV_PLAN_UNIT_INTS + lane) : 0;
  const int32_t agent = r / a.hkv / a.chunks;
  return lane == 0 ? __ldg(a.seq_lens + agent) : 0;
}

// Field `lane` of unit r's descriptor (lanes >= kUnitInts: 0) and, in `next`, the CTA's unit
// after it (-1: none).  Every lane checks the whole record (an invalid unit becomes empty and
// raises kDevBadArg); lanes of the per-agent fields issue their loads here and do not wait.
__device__ __forceinline__ int32_t unit_field(const DecodeArgs& a, int32_t r, int32_t raw, int lane, int32_t& next) {
  if (r < 0) {
    next = -1;
    return lane == kUfEnd ? 1 : 0;
  }
  int32_t p0, p1, na, h, slot, ag[kMaxGroup];
  if (a.units) {
    p0 = __shfl_sync(0xffffffffu, raw, 0);
    p1 = __shfl_sync(0xffffffffu, raw, 1);
    na = __shfl_sync(0xffffffffu, raw, 2);
    h = __shfl_sync(0xffffffffu, raw, 3);
    slot = __shfl_sync(0xffffffffu, raw, 4);
    next = __shfl_sync(0xffffffffu, raw, 5);
#pragma unroll
    for (int x = 0; x < kMaxGroup; ++x) ag[x] = __shfl_sync(0xffffffffu, raw, 6 + x);
    bool bad = false;
    if (na != 1 && na != 2 && na != 4) {  // the value products stack the slots of 1, 2 or 4 agents
      bad = true;
      na = 1;
    }
    if (slot < 0 || slot + na > a.n_slots) {
      bad = true;
      slot = -1;  // empty: reads nothing, writes nothing
    }
    if (next != -1 && (next <= r || next >= a.n_units)) {  // links only go forward
      bad = true;
      next = -1;
    }
    if (bad) {
      if (lane == 0) flag_status(a.status, kDevBadArg);
      p1 = p0;
    }
  } else {
    const int32_t item = r / a.hkv, agent = item / a.chunks, c = item % a.chunks;
    h = r - item * a.hkv;
    const int32_t L = min(__shfl_sync(0xffffffffu, raw, 0), a.max_seq_len);
    p0 = c * a.chunk_pages;
    p1 = min(p0 + a.chunk_pages, (L + kPage - 1) / kPage);
    na = 1;
    slot = item;
#pragma unroll
    for (int x = 0; x < kMaxGroup; ++x) ag[x] = agent;
    next = r + (int32_t)gridDim.x < a.n_units ? r + (int32_t)gridDim.x : -1;
  }
  bool bad = (uint32_t)h >= (uint32_t)a.hkv || p0 < 0 || p1 > a.pt_stride;
#pragma unroll
  for (int x = 0; x < kMaxGroup; ++x) bad |= (uint32_t)ag[x] >= (uint32_t)a.n_agents;
  if (bad) {
    if (lane == 0) flag_status(a.status, kDevBadArg);
    h = 0;
    p0 = p1 = 0;
#pragma unroll
    for (int x = 0; x < kMaxGroup; ++x) ag[x] = 0;
  }
  if (p1 < p0) p1 = p0;
  const int x = (lane - kUfAgent) & 3;  // agent of the per-agent field lanes
  int32_t agx = ag[0];
#pragma unroll
  for (int i = 1; i < kMaxGroup; ++i)
    if (x == i) agx = ag[i];
  switch (lane < kUfAgent ? lane : kUfAgent + 4 * ((lane - kUfAgent) >> 2)) {
    case kUfP0: return p0;
    case kUfP1: return p1;
    case kUfNa: return na;
    case kUfH: return h;
    case kUfSlot: return slot;
    case kUfEnd: return 0;
    case kUfAgent: return agx;
    case kUfL: return x < na ? __ldg(a.seq_lens + agx) : 0;  // clipped and checked at publication
    case kUfPos: return __ldg(a.positions + agx);
    case kUfAdapter: return a.adapter_ids ? __ldg(a.adapter_ids + agx) : agx;
    case kUfHole: {
      if (!a.holes) return 0;
      const int32_t hs = __ldg(a.holes + 2 * agx), hn = __ldg(a.holes + 2 * agx + 1);
      if (hn == 0) return 0;
      if (hn < 0 || hn >= kPage || hs < 0 || hs > (1 << 26)) {
        flag_status(a.status, kDevBadArg);
        return 0;
      }
      return hs * kPage + hn;
    }
    default: return 0;
  }
}

// Descriptor field at publication, when the agents' loads have landed: each agent's length
// clipped to max_seq_len, after the checks on it and on its query position.
__device__ __forceinline__ int32_t unit_finish(const DecodeArgs& a, int32_t v, int lane) {
  const int32_t pos = __shfl_down_sync(0xffffffffu, v, kUfPos - kUfL);  // lane kUfL + x: agent x's position
  const int32_t na = __shfl_sync(0xffffffffu, v, kUfNa);
  const int32_t end = __shfl_sync(0xffffffffu, v, kUfEnd);
  if (lane < kUfL || lane >= kUfL + kMaxGroup || end) return v;
  if (lane - kUfL >= na) return 0;
  if (v < 1 || v > a.max_seq_len || pos < 0 || pos >= v) flag_status(a.status, kDevBadArg);
  return min(v, a.max_seq_len);
}

// Page copies of one block, by groups of 8 lanes: group q holds the ids of the block's nvp
// (<= 8) pages in its lanes 8 q + p.  A base tile keeps its rows in two 2048-byte halves (128
// bytes a row), a residual tile in one (32 bytes a row).  When rows < 16 only the first rows
// of the last page are copied.

// Bytes the copies of one group deliver.
__device__ __forceinline__ uint32_t tile_bytes(bool base, int nvp, int rows) {
  const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
  return rows < kPage ? (uint32_t)(nvp - 1) * tile + (base ? 2u : 1u) * (uint32_t)rows * rb : (uint32_t)nvp * tile;
}

// Zero the rows of the last page that are not copied (rows past every sequence may never have
// been written, and a zero probability must not meet a NaN).  Lane p of the group.
__device__ __forceinline__ void zero_tail(bool base, int nvp, int rows, uint8_t* dst, int p) {
  if (rows >= kPage) return;
  const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
  uint8_t* t = dst + (nvp - 1) * tile;
  const uint32_t half = base ? 2048u : tile;  // bytes per half
  for (uint32_t o = rows * rb + 16 * p; o < half; o += 16 * 8) {
    *reinterpret_cast<uint4*>(t + o) = make_uint4(0u, 0u, 0u, 0u);
    if (base) *reinterpret_cast<uint4*>(t + 2048 + o) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Lane p of a group issues its share of the copies, with no warp-wide operation: consecutive
// ids (one_run) as one bulk copy from the group's first lane, otherwise one copy per page; the
// lane holding a partial last page copies its rows.  The barrier's expected bytes are raised
// by the caller in the same arrival that completes its count.
__device__ __forceinline__ void copy_tiles(const uint8_t* pool, bool base, int32_t id, int nvp, int rows, uint8_t* dst,
                                           uint64_t* bar, bool one_run, int p) {
  const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
  const int full = rows < kPage ? nvp - 1 : nvp;  // pages copied whole
  if (one_run) {
    if (p == 0 && full > 0) bulk_g2s(dst, pool + (int64_t)id * tile, full * tile, bar);
  } else if (p < full) {
    bulk_g2s(dst + p * tile, pool + (int64_t)id * tile, tile, bar);
  }
  if (full < nvp && rows > 0 && p == full) {
    const uint8_t* src = pool + (int64_t)id * tile;
    bulk_g2s(dst + full * tile, src, rows * rb, bar);
    if (base) bulk_g2s(dst + full * tile + 2048, src + 2048, rows * rb, bar);
  }
}

// Every wait of this kernel hints the hardware to suspend the waiting thread for up to 1 us
// per poll (it wakes as soon as the phase completes), so waiting warps leave the issue slots to
// the working ones (measured: 1-1.5 % faster than polls without the hint).
constexpr uint32_t kSuspendNs = 1000;

// Bounded wait for a phase (acquire), suspending between polls.
__device__ __forceinline__ bool mbar_wait_s(uint64_t* bar, uint32_t parity, uint32_t* status) {
#pragma unroll 1
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait_for(bar, parity, kSuspendNs)) return true;
  flag_status(status, kDevTimeout);
  return false;
}

// Wait for a phase completed by a tensor-core commit (the waiter orders its tensor-memory
// accesses with tcgen05.fence::after_thread_sync, so no memory acquire is needed).
__device__ __forceinline__ bool mbar_wait_tc(uint64_t* bar, uint32_t parity, uint32_t* status) {
#pragma unroll 1
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.relaxed.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
  }
  flag_status(status, kDevTimeout);
  return false;
}

// Maximum over the 32 lanes of a warp.
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// The reference maximum of a (unit, agent, query head) before any visible key: a finite floor
// rather than -inf, so that s - m is never -inf - (-inf) and needs no guard.  The first visible
// key always passes it by 2^8 and sets the reference; the epilogue reports the floor as -inf.
constexpr float kNoMax = -3.4028234663852886e38f;

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
  int32_t* s_lp = reinterpret_cast<int32_t*>(smem + 1280);  // [4 warps][4 agents][2] visible limit, hole start
  int32_t* s_units = reinterpret_cast<int32_t*>(smem + kOffUnits);  // [2][kUnitInts] unit descriptors
  int32_t* s_lh = reinterpret_cast<int32_t*>(smem + kOffHoles);      // [4 warps][4 agents] hole end

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t count = 1;  // a single arrival: the producer's expect_tx or one MMA commit
      if (i == kKEmpty0 || i == kKEmpty1 || i == kUFree0 || i == kUFree1 || i == kKFFull0 || i == kKFFull1)
        count = kRopeWarps;  // one arrival per RoPE warp
      if ((i >= kSFree0 && i <= kSFree2) || i == kPFull0 || i == kPFull1 || i == kRed0 || i == kRed1 ||
          i == kEpiDone)
        count = 4;  // one arrival per softmax warp
      if (i == kUnitFree0 || i == kUnitFree1) count = kThreads / 32 - 1;  // every warp but the producer
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

  // Unit k of this CTA as published by the producer: wait for its descriptor, and release
  // the ring slot once the caller has copied what it needs (`take`).
  auto unit_wait = [&](int k) { return mbar_wait_s(&bars[kUnitReady0 + (k & 1)], (k >> 1) & 1, a.status); };
  auto unit_at = [&](int k, int f) -> int32_t { return s_units[(k & 1) * kUnitInts + f]; };
  auto unit_release = [&](int k) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kUnitFree0 + (k & 1)]);
  };
  auto blocks_of = [](int32_t p0, int32_t p1) { return (p1 - p0 + kBlockPages - 1) / kBlockPages; };

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    // Describes the units in the ring (descriptors built two ahead, so that the loads behind
    // one land while earlier units run) and copies, block by block: the K tiles, each agent's
    // k_res tiles as soon as that agent's slot (four steps back) is free, then the V tiles
    // with every agent's v_res tiles.  Every wait is for a buffer's previous user.  Page ids
    // come one per lane (lane p < 8 the base page p, lane 8 a + p the residual page p of agent
    // a) and are requested two blocks ahead.
    const int pg = lane & 7, ag = lane >> 3;
    int32_t r_nxt;
    const int32_t r0 = first_unit(a);
    int32_t cur = unit_field(a, r0, unit_raw(a, r0, lane), lane, r_nxt);  // next descriptor to publish
    int32_t raw_nxt = unit_raw(a, r_nxt, lane);                            // raw record of the one after
    int n_pub = 0;
    bool ok = true;
    // publish `cur` as unit n_pub once its ring slot is free; build the next descriptor
    auto publish = [&]() -> int32_t {
      if (n_pub >= 2) ok = ok && mbar_wait_s(&bars[kUnitFree0 + (n_pub & 1)], ((n_pub >> 1) - 1) & 1, a.status);
      const int32_t v = unit_finish(a, cur, lane);
      if (lane < kUnitInts) s_units[(n_pub & 1) * kUnitInts + lane] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kUnitReady0 + (n_pub & 1)]);
      ++n_pub;
      if (__shfl_sync(0xffffffffu, v, kUfEnd) == 0) {
        const int32_t r = r_nxt;
        cur = unit_field(a, r, raw_nxt, lane, r_nxt);
        raw_nxt = unit_raw(a, r_nxt, lane);
      }
      return v;
    };
    struct Blk {  // what the copies of one block need
      int32_t bid, bx, rid, h, na, pbase, nvp, Lmax, Lx;
    };
    int kbl = 0, knb = 0;  // the cursor: next block within its unit, and the unit's blocks
    bool ended = false;
    int32_t kp0 = 0, kp1 = 0, kna = 1, kh = 0, kag0 = 0, kagx = 0, kLx = 0, kLmax = 0;
    // the cursor's next block into x, its page ids requested (not waited for); false at the end
    auto next_block = [&](Blk& x) -> bool {
      while (kbl >= knb) {
        if (ended || !ok) return false;
        const int32_t d = publish();
        if (__shfl_sync(0xffffffffu, d, kUfEnd) != 0) {
          ended = true;
          return false;
        }
        kp0 = __shfl_sync(0xffffffffu, d, kUfP0);
        kp1 = __shfl_sync(0xffffffffu, d, kUfP1);
        kna = __shfl_sync(0xffffffffu, d, kUfNa);
        kh = __shfl_sync(0xffffffffu, d, kUfH);
        kag0 = __shfl_sync(0xffffffffu, d, kUfAgent);
        kagx = __shfl_sync(0xffffffffu, d, kUfAgent + (ag & 3));
        kLx = __shfl_sync(0xffffffffu, d, kUfL + (ag & 3));
        if (ag >= kna) kLx = 0;
        kLmax = kLx;  // rows at or past the longest sequence of the group are never read as data
#pragma unroll
        for (int o = 8; o < 32; o <<= 1) kLmax = max(kLmax, __shfl_xor_sync(0xffffffffu, kLmax, o));
        knb = blocks_of(kp0, kp1);
        kbl = 0;
      }
      x.pbase = kp0 + kbl * kBlockPages;
      x.nvp = min(kBlockPages, kp1 - x.pbase);
      x.h = kh;
      x.na = kna;
      x.Lmax = kLmax;
      x.Lx = kLx;
      x.bid = x.bx = x.rid = 0;
      if (lane < x.nvp) x.bid = a.bpt[(int64_t)kag0 * a.pt_stride + x.pbase + lane];
      if (ag < kna && pg < x.nvp) {
        x.rid = a.rpt[(int64_t)kagx * a.pt_stride + x.pbase + pg];
        if (ag > 0) x.bx = a.bpt[(int64_t)kagx * a.pt_stride + x.pbase + pg];  // the other agents' base pages
      }
      ++kbl;
      return true;
    };
    Blk nx{}, nx2{};  // the next two blocks
    bool more = next_block(nx);
    bool more2 = more && next_block(nx2);
    int g = 0, kn = 0;  // blocks copied, k_res steps copied
    while (ok && more) {
      Blk b = nx;
      nx = nx2;
      more = more2;
      if (more2) more2 = next_block(nx2);  // the ids of the block after next go out now
      // The group shares its base pages: the first agent's ids serve every agent.  A plan built
      // before a copy-on-write split, a commit or an append that changed an agent's pages no
      // longer matches the page tables: reported (the first agent's pages are read).
      const int32_t b0 = __shfl_sync(0xffffffffu, b.bid, pg);  // the first agent's page pg
      if (ag > 0 && ag < b.na && pg < b.nvp && b.bx != b0) flag_status(a.status, kDevBadArg);
      if ((uint32_t)b.bid >= (uint32_t)a.num_base_pages) {
        flag_status(a.status, kDevBadPage);
        b.bid = 0;
      }
      if ((uint32_t)b.rid >= (uint32_t)a.num_res_pages) {
        flag_status(a.status, kDevBadPage);
        b.rid = 0;
      }
      const int32_t pb = __shfl_up_sync(0xffffffffu, b.bid, 1), pr = __shfl_up_sync(0xffffffffu, b.rid, 1);
      const bool brun = __ballot_sync(0xffffffffu, lane < 8 && pg > 0 && pg < b.nvp && b.bid != pb + 1) == 0;
      const bool rrun = ((__ballot_sync(0xffffffffu, pg > 0 && pg < b.nvp && b.rid != pr + 1) >> (lane & ~7)) & 0xffu) == 0;
      // K tiles
      if (g >= 2 && !(ok = mbar_wait_s(&bars[kKEmpty0 + (g & 1)], ((g >> 1) - 1) & 1, a.status))) break;
      uint64_t* kbar = &bars[kKFull0 + (g & 1)];
      if (lane == 0) mbar_arrive_expect_tx(kbar, tile_bytes(true, b.nvp, kPage));
      if (lane < 8)
        copy_tiles(a.k_base + (int64_t)b.h * a.num_base_pages * kBaseTile, true, b.bid, b.nvp, kPage,
                   smem + kOffK + (g & 1) * kBlockTiles, kbar, brun, pg);
      // each agent's k_res tiles, into the slot of its (block, agent) step
      for (int x = 0; x < b.na && ok; ++x) {
        const int n = kn + x, kslot = n & 3;
        if (n >= kResSlots && !(ok = mbar_wait_s(&bars[kKrEmpty0 + kslot], ((n >> 2) - 1) & 1, a.status))) break;
        uint64_t* rbar = &bars[kKrFull0 + kslot];
        if (lane == 8 * x) mbar_arrive_expect_tx(rbar, tile_bytes(false, b.nvp, kPage));
        if (ag == x) copy_tiles(a.k_res, false, b.rid, b.nvp, kPage, smem + kOffKr + kslot * kResSlotBytes, rbar, rrun, pg);
      }
      if (!ok) break;
      kn += b.na;
      // V tiles and every agent's v_res tiles, on one barrier (released by the block's value
      // products); one arrival raises the bytes of every group
      if (g >= 2 && !(ok = mbar_wait_s(&bars[kVEmpty0 + (g & 1)], ((g >> 1) - 1) & 1, a.status))) break;
      uint64_t* vbar = &bars[kVFull0 + (g & 1)];
      const int last = (b.pbase + b.nvp - 1) * kPage;  // first key of the block's last page
      const int vrows = min(kPage, max(0, b.Lmax - last));
      const int rrows = min(kPage, max(0, b.Lx - last));  // this lane group's agent
      uint8_t* vdst = smem + kOffV + (g & 1) * kBlockTiles;
      uint8_t* rdst = smem + kOffVr + (g & 1) * kVrGroupBytes + (4 - b.na + ag) * kResSlotBytes;
      const bool ract = ag < b.na;
      if (__any_sync(0xffffffffu, (lane < 8 && vrows < kPage) || (ract && rrows < kPage))) {
        if (lane < 8) zero_tail(true, b.nvp, vrows, vdst, pg);
        if (ract) zero_tail(false, b.nvp, rrows, rdst, pg);
        tc::fence_proxy_async();
        __syncwarp();
      }
      uint32_t bytes = ract && pg == 0 ? tile_bytes(false, b.nvp, rrows) : 0u;
      bytes += __shfl_xor_sync(0xffffffffu, bytes, 8);
      bytes += __shfl_xor_sync(0xffffffffu, bytes, 16);
      if (lane == 0) mbar_arrive_expect_tx(vbar, bytes + tile_bytes(true, b.nvp, vrows));
      if (lane < 8)
        copy_tiles(a.v_base + (int64_t)b.h * a.num_base_pages * kBaseTile, true, b.bid, b.nvp, vrows, vdst, vbar, brun, pg);
      if (ract) copy_tiles(a.v_res, false, b.rid, b.nvp, rrows, rdst, vbar, rrun, pg);
      ++g;
    }
    // never leave with copies in flight: the last phase of every barrier written to
    for (int b = max(0, g - 2); b < g; ++b) {
      mbar_wait_s(&bars[kKFull0 + (b & 1)], (b >> 1) & 1, a.status);
      mbar_wait_s(&bars[kVFull0 + (b & 1)], (b >> 1) & 1, a.status);
    }
    for (int n = max(0, kn - kResSlots); n < kn; ++n) mbar_wait_s(&bars[kKrFull0 + (n & 3)], (n >> 2) & 1, a.status);
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
    for (int k = 0; ok; ++k) {
      if (!unit_wait(k)) break;
      const int32_t p0 = unit_at(k, kUfP0), p1 = unit_at(k, kUfP1), na = unit_at(k, kUfNa), h = unit_at(k, kUfH);
      const bool end = unit_at(k, kUfEnd) != 0;
      int32_t adapter = unit_at(k, kUfAdapter + (lane & 3));
      unit_release(k);
      if (end) break;
      const int N = blocks_of(p0, p1) * na;
      if ((lane & 3) < na && (uint32_t)adapter >= (uint32_t)a.n_adapters) {
        flag_status(a.status, kDevBadArg);
        adapter = 0;
      }
      if (k > 0) {  // every U of the previous unit is done with B_k
        if (lane == 0) {
          tc::commit(&bars[kUUnit]);
          ok = mbar_wait_s(&bars[kUUnit], (k - 1) & 1, a.status);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      for (int x = 0; x < na; ++x) {
        int32_t ad = __shfl_sync(0xffffffffu, adapter, x);
        if ((uint32_t)ad >= (uint32_t)a.n_adapters) ad = 0;
        const __nv_bfloat16* B = a.B_k + (int64_t)ad * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // 16 ranks x 16 chunks of 8 d
          const int c = lane + 32 * i, r = c >> 4, ch = c & 15;
          v[i] = *reinterpret_cast<const uint4*>(B + (int64_t)r * a.hkv * kHeadDim + ch * 8);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = lane + 32 * i, r = c >> 4, ch = c & 15;
          *reinterpret_cast<uint4*>(smem + kOffBk + x * 4096 + base_off(r, ch * 8)) = v[i];
        }
      }
      tc::fence_proxy_async();
      __syncwarp();
      for (int n = 0, ai = 0; n < N && ok; ++n) {
        const int m = gn + n;
        ok = mbar_wait_s(&bars[kKrFull0 + (m & 3)], (m >> 2) & 1, a.status) &&
             (m < 2 || mbar_wait_s(&bars[kUFree0 + (m & 1)], ((m >> 1) - 1) & 1, a.status));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after();
        const uint64_t dk = dKr + (m & 3) * (kResSlotBytes >> 4), db = dBk + ai * (4096 >> 4);
        const uint32_t du = tm + kTmU + 128 * (m & 1);
        if (tc::elect_one()) {
          tc::mma_ss(du, dk, db, idU, 0);
          tc::commit(&bars[kUFull0 + (m & 1)]);
          tc::commit(&bars[kKrEmpty0 + (m & 3)]);
        }
        __syncwarp();
        if (++ai == na) ai = 0;
      }
      gn += N;
    }
    if (lane == 0) {
      tc::commit(&bars[kMmaDone]);  // never leave with MMAs in flight
      mbar_wait_s(&bars[kMmaDone], 0, a.status);
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
    for (int k = 0; ok; ++k) {
      if (!unit_wait(k)) break;
      const int32_t p0 = unit_at(k, kUfP0), p1 = unit_at(k, kUfP1), na = unit_at(k, kUfNa), h = unit_at(k, kUfH);
      const bool end = unit_at(k, kUfEnd) != 0;
      const int32_t agent_l = unit_at(k, kUfAgent + (lane & 3));
      unit_release(k);
      if (end) break;
      const int N = blocks_of(p0, p1) * na;
      if (k > 0) {  // every S of the previous unit is done with Q^T
        if (lane == 0) {
          tc::commit(&bars[kSUnit]);
          ok = mbar_wait_s(&bars[kSUnit], (k - 1) & 1, a.status);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      uint4 v[kMaxGroup][4];
#pragma unroll
      for (int x = 0; x < kMaxGroup; ++x) {
        const int32_t agent = __shfl_sync(0xffffffffu, agent_l, x);
#pragma unroll
        for (int i = 0; i < 4; ++i) {  // 8 query-head rows x 16 chunks of 8 d
          const int c = lane + 32 * i, g = c >> 4, ch = c & 15;
          v[x][i] = make_uint4(0u, 0u, 0u, 0u);
          if (x < na && g < G)
            v[x][i] = *reinterpret_cast<const uint4*>(a.q + ((int64_t)agent * a.hkv * G + (int64_t)h * G + g) * kHeadDim +
                                                      ch * 8);
        }
      }
#pragma unroll
      for (int x = 0; x < kMaxGroup; ++x)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i, g = c >> 4, ch = c & 15;
          if (x < na) *reinterpret_cast<uint4*>(smem + kOffQ + x * 2048 + tc::sw128_off(8, g, ch * 8)) = v[x][i];
        }
      tc::fence_proxy_async();
      __syncwarp();
      int sr = gn % kSRing, sp = (gn / kSRing) & 1;  // S ring slot and its phase of step gn
      for (int n = 0, ai = 0; n < N && ok; ++n) {
        const int m = gn + n;
        const int kr = m & 1;
        ok = mbar_wait_s(&bars[kKFFull0 + kr], (m >> 1) & 1, a.status) &&
             (m < kSRing || mbar_wait_s(&bars[kSFree0 + sr], sp ^ 1, a.status));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after();
        const uint32_t q = kOffQ + ai * 2048;  // the two 64-column halves of Q^T at q, q + 1024
        const uint64_t dq0 = tc::smem_desc(sBase + q, 16, kOffQZero - q, tc::kSwizzle128B);
        const uint64_t dq1 = tc::smem_desc(sBase + q + 1024, 16, kOffQZero - q - 1024, tc::kSwizzle128B);
        const uint32_t dS = tm + kTmS + 16 * sr, aK = tm + kTmKF + 64 * kr;
        if (tc::elect_one()) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)  // K = 16 per step: 8 TMEM columns of A, 32 bytes of B
            tc::mma_ts(dS, aK + 8 * ks, (ks < 4 ? dq0 : dq1) + 2 * (ks & 3), idS, ks > 0);
          tc::commit(&bars[kSFull0 + sr]);
          tc::commit(&bars[kKFFree0 + kr]);
        }
        __syncwarp();
        if (++ai == na) ai = 0;
        if (++sr == kSRing) {
          sr = 0;
          sp ^= 1;
        }
      }
      gn += N;
    }
    if (lane == 0) {
      tc::commit(&bars[kSDone]);
      mbar_wait_s(&bars[kSDone], 0, a.status);
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
    for (int k = 0; ok; ++k) {
      if (!unit_wait(k)) break;
      const int32_t p0 = unit_at(k, kUfP0), p1 = unit_at(k, kUfP1), na = unit_at(k, kUfNa);
      // The key in slot j sits at position j, or j - hole length past the agent's hole.  Agents
      // that share a page past a hole have the same hole (it came with the pages), and a slot in
      // the page of a hole is at its own index for every agent that sees it, so the first
      // agent's hole gives the rotation position of every visible key of the item.
      const int32_t hc0 = unit_at(k, kUfHole);
      const bool end = unit_at(k, kUfEnd) != 0;
      unit_release(k);
      if (end) break;
      const int32_t hend = (hc0 >> 4) + (hc0 & 15), hn0 = hc0 & 15;
      const int N = blocks_of(p0, p1) * na;
      for (int n = 0, b = 0, ai = 0; n < N && ok; ++n, ai = ai + 1 == na ? 0 : ai + 1, b += ai == 0) {
        const int g = gb + b, m = gn + n;  // global block and step
        const int stage = g & 1;
        const int pbase = p0 + b * kBlockPages;
        const int j = pbase * kPage + row;
        if (ai == 0) {
          // chunk c = 32 hf + 16 cc holds frequency groups m = c/2 .. c/2 + 7: the 32-byte group
          // blocks c/8 and c/8 + 1 of position jr (rope_off(jr, 4 u) for block u)
          const int kp = (hn0 != 0 && j >= hend) ? j - hn0 : j;
          const int jr = kp < a.rope_positions ? kp : 0;
          const uint8_t* rrow = a.rope + rope_off(jr, 0);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int uu = 0; uu < 2; ++uu) {
              const int un = 4 * hf + 2 * cc + uu;
              rp[cc][2 * uu] = __ldg(reinterpret_cast<const uint4*>(rrow + un * 512));
              rp[cc][2 * uu + 1] = __ldg(reinterpret_cast<const uint4*>(rrow + un * 512 + 16));
            }
          ok = mbar_wait_s(&bars[kKFull0 + stage], (g >> 1) & 1, a.status);
          if (!ok) break;
        }
        // U of this step, read out at once (as bf16 pairs) so that its buffer frees early
        ok = mbar_wait_tc(&bars[kUFull0 + (m & 1)], (m >> 1) & 1, a.status);
        if (!ok) break;
        tc::fence_after();
        uint32_t ul[2][8], uh[2][8];  // [chunk][pair]: U columns (c + 2 i, c + 2 i + 1) and + 64
        {
          uint32_t lo[2][16], hi[2][16];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 32 * hf + 16 * cc;
            tc::ld16(tl + kTmU + 128 * (m & 1) + c, lo[cc]);
            tc::ld16(tl + kTmU + 128 * (m & 1) + 64 + c, hi[cc]);
          }
          tc::wait_ld();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              ul[cc][i] = pack_bf16(__uint_as_float(lo[cc][2 * i]), __uint_as_float(lo[cc][2 * i + 1]));
              uh[cc][i] = pack_bf16(__uint_as_float(hi[cc][2 * i]), __uint_as_float(hi[cc][2 * i + 1]));
            }
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kUFree0 + (m & 1)]);
        const int kr = m & 1;
        if (m >= kKfRing && !mbar_wait_tc(&bars[kKFFree0 + kr], ((m >> 1) - 1) & 1, a.status)) {
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
            // K = Kb + RoPE_j(U) in two fused multiply-adds per bf16x2 pair: Kb - U_hi sin,
            // then + U_lo cos (and Kb + U_lo sin, then + U_hi cos), each rounded to bf16 at K's
            // scale (two roundings of K instead of one: measured rel_l2 3.4e-3 against 2.9e-3, for
            // a third fewer rotation instructions)
            const __nv_bfloat162 C = *reinterpret_cast<const __nv_bfloat162*>(&cw);
            const __nv_bfloat162 S = *reinterpret_cast<const __nv_bfloat162*>(&sw);
            const __nv_bfloat162 UL = *reinterpret_cast<const __nv_bfloat162*>(&ul[cc][i2]);
            const __nv_bfloat162 UH = *reinterpret_cast<const __nv_bfloat162*>(&uh[cc][i2]);
            const __nv_bfloat162 kl2 =
                __hfma2(UL, C, __hfma2(__hneg2(UH), S, *reinterpret_cast<const __nv_bfloat162*>(&klw[i2])));
            const __nv_bfloat162 kh2 = __hfma2(UH, C, __hfma2(UL, S, *reinterpret_cast<const __nv_bfloat162*>(&khw[i2])));
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
      gb += blocks_of(p0, p1);
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
    const uint32_t sBase = smem_u32(smem);
    const uint64_t dV = tc::smem_desc(sBase + kOffV, 2048, 1024, tc::kSwizzle128B);
    const uint64_t dP = tc::smem_desc(sBase + kOffP, 4096, 256, tc::kSwizzle32B);
    int gb = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!unit_wait(k)) break;
      const int32_t p0 = unit_at(k, kUfP0), p1 = unit_at(k, kUfP1), na = unit_at(k, kUfNa);
      const bool end = unit_at(k, kUfEnd) != 0;
      unit_release(k);
      if (end) break;
      const int nb = blocks_of(p0, p1);
      const uint32_t idV = tc::idesc_bf16(128, na > 2 ? 32 : 16, 1, 1);
      const uint64_t dR =
          tc::smem_desc(sBase + kOffVr + (4 - na) * kResSlotBytes, kResSlotBytes, 256, tc::kSwizzle32B);
      if (k > 0) ok = __all_sync(0xffffffffu, mbar_wait_s(&bars[kEpiDone], (k - 1) & 1, a.status));
      for (int b = 0; b < nb && ok; ++b) {
        const int g = gb + b;
        ok = mbar_wait_s(&bars[kVFull0 + (g & 1)], (g >> 1) & 1, a.status) &&
             mbar_wait_s(&bars[kPFull0 + (g & 1)], (g >> 1) & 1, a.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc::fence_after();
        const int nvp = min(kBlockPages, p1 - (p0 + b * kBlockPages));
        const uint64_t dv = dV + (g & 1) * (kBlockTiles >> 4), dp = dP + (g & 1) * (8192 >> 4);
        const uint64_t dr = dR + (g & 1) * (kVrGroupBytes >> 4);  // 8 atoms of 16 rows, 4 KB apart
        const uint32_t acc0 = b > 0;
        if (tc::elect_one()) {
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
        __syncwarp();
      }
      gb += nb;
    }
    if (tc::elect_one()) {
      tc::commit(&bars[kValDone]);
      mbar_wait_s(&bars[kValDone], 0, a.status);
    }
    __syncwarp();
  } else {
    // ------------------------------ softmax group ------------------------------
    const int sw_ = warp & 3;
    const int row = 32 * sw_ + lane;  // key row of the block == TMEM lane (and d row of O^T)
    const uint32_t tl = tm + ((uint32_t)(32 * sw_) << 16);
    float* mref = s_mref + sw_ * (kMaxGroup * 8);  // this warp's copy (all four evolve identically)
    int32_t* lp = s_lp + sw_ * (kMaxGroup * 2);    // this warp's copy of each agent's (visible limit, hole start)
    int32_t* lh = s_lh + sw_ * kMaxGroup;          // and of each agent's hole end
    // query head whose reference maximum this lane publishes after a rescale, and the publishing lanes
    const int gl = kG == 8 ? lane >> 2 : lane >> 3;
    const bool publisher = kG == 8 ? (lane & 3) == 0 : (lane & 7) == 0;
    int gb = 0, gn = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!unit_wait(k)) break;
      const int32_t p0 = unit_at(k, kUfP0), p1 = unit_at(k, kUfP1), na = unit_at(k, kUfNa), h = unit_at(k, kUfH);
      const int32_t slot_base = unit_at(k, kUfSlot);
      const bool end = unit_at(k, kUfEnd) != 0;
      __syncwarp();
      mref[lane] = kNoMax;  // 4 agents x 8 query heads
      if (lane < kMaxGroup) {
        // Agent `lane`'s visible slots: j < lim, outside its hole [hlo, hhi).  The key in slot j
        // sits at position j, or j - hole length past the hole, so a query at position pos sees
        // slot j up to pos (pos before the hole) or pos + hole length (pos past it); slots past
        // the agent's length or the unit's pages are never visible.
        const int32_t L = unit_at(k, kUfL + lane), pos = unit_at(k, kUfPos + lane);  // L: 0 past the unit's agents
        const int32_t hc = unit_at(k, kUfHole + lane), hs = hc >> 4, hn = hc & 15;
        const int32_t last = (hn != 0 && pos >= hs) ? pos + hn : pos;  // the query's own slot
        lp[2 * lane] = min(min(L, p1 * kPage), last + 1);
        lp[2 * lane + 1] = hs;
        lh[lane] = hs + hn;
      }
      unit_release(k);
      if (end) break;
      const int nb = blocks_of(p0, p1), N = nb * na;
      int sr = gn % kSRing, sp = (gn / kSRing) & 1;  // S ring slot and its phase of step gn
      for (int n = 0, b = 0, ai = 0; n < N && ok;
           ++n, ai = ai + 1 == na ? 0 : ai + 1, b += ai == 0, sp ^= sr + 1 == kSRing, sr = sr + 1 == kSRing ? 0 : sr + 1) {
        const int g = gb + b, m = gn + n;  // global block and step
        const int pbase = p0 + b * kBlockPages;
        const int j = pbase * kPage + row;
        const int2 lim_lo = reinterpret_cast<const int2*>(lp)[ai];  // (visible limit, hole start)
        const bool vis = j < lim_lo.x && (j < lim_lo.y || j >= lh[ai]);
        ok = mbar_wait_tc(&bars[kSFull0 + sr], sp, a.status);
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
        // max over the warp's keys of each query head, stored by one lane as float4s
        float* red = s_red + (m & 1) * 32;
        {
          float wq[kG];
#pragma unroll
          for (int q = 0; q < kG; ++q) wq[q] = warp_max(sc[q]);
          if (lane == 0) {
            float4* r4 = reinterpret_cast<float4*>(red + sw_ * kG);
            r4[0] = make_float4(wq[0], wq[1], wq[2], wq[3]);
            if constexpr (kG == 8) r4[1] = make_float4(wq[4 % kG], wq[5 % kG], wq[6 % kG], wq[7 % kG]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kRed0 + (m & 1)]);
        // while the other warps' maxima come in: probabilities against the current reference
        // (a masked score is -inf and the reference is finite, so 2^(s - m) = 0 needs no mask)
        float mr[kG], ps[kG];
        {
          const float4* m4 = reinterpret_cast<const float4*>(mref + ai * 8);
          const float4 x0 = m4[0];
          mr[0] = x0.x;
          mr[1] = x0.y;
          mr[2] = x0.z;
          mr[3] = x0.w;
          if constexpr (kG == 8) {
            const float4 x1 = m4[1];
            mr[4 % kG] = x1.x;
            mr[5 % kG] = x1.y;
            mr[6 % kG] = x1.z;
            mr[7 % kG] = x1.w;
          }
        }
#pragma unroll
        for (int q = 0; q < kG; ++q) ps[q] = ex2(sc[q] - mr[q]);
        ok = mbar_wait_s(&bars[kRed0 + (m & 1)], (m >> 1) & 1, a.status);
        if (!ok) break;
        // lazy rescale: keep the reference maximum unless the block maximum passes it by 2^8
        float bm[kG];
        bool need_any = false;
        {
          float4 x[4][2];  // the four warps' maxima, read as float4s
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            x[w][0] = reinterpret_cast<const float4*>(red + w * kG)[0];
            if constexpr (kG == 8) x[w][1] = reinterpret_cast<const float4*>(red + w * kG)[1];
          }
#pragma unroll
          for (int q = 0; q < kG; ++q) {
            float v[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const float4 y = x[w][q >> 2];
              v[w] = (q & 3) == 0 ? y.x : (q & 3) == 1 ? y.y : (q & 3) == 2 ? y.z : y.w;
            }
            bm[q] = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
            need_any |= bm[q] > mr[q] + 8.f;  // heads past G: -inf scores, never a rescale
          }
        }
        if (need_any) {  // uniform across the group: every warp saw the same maxima
          float alpha[kG];
#pragma unroll
          for (int q = 0; q < kG; ++q) {
            const bool need = bm[q] > mr[q] + 8.f;
            // from the floor kNoMax, alpha = 0: O and R hold only zero probabilities until then
            alpha[q] = need ? ex2(mr[q] - bm[q]) : 1.f;
            if (need) mr[q] = bm[q];
          }
          float ml = mr[0];
#pragma unroll
          for (int q = 1; q < kG; ++q)
            if (gl == q) ml = mr[q];
          __syncwarp();
          if (publisher) mref[ai * 8 + gl] = ml;
#pragma unroll
          for (int q = 0; q < kG; ++q) ps[q] = ex2(sc[q] - mr[q]);
          if (b > 0) {
            // O^T and R are stable once the value products of block g - 1 are done (one barrier
            // per block parity, so a wait is never more than one phase ahead of the barrier)
            ok = mbar_wait_s(&bars[kODone0 + ((g - 1) & 1)], ((g - 1) >> 1) & 1, a.status);
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
        if (ai == 0 && g >= 2) ok = mbar_wait_s(&bars[kPFree0 + (g & 1)], ((g >> 1) - 1) & 1, a.status);
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
      if (nb > 0) ok = mbar_wait_s(&bars[kODone0 + (glast & 1)], (glast >> 1) & 1, a.status);
      tc::fence_after();
      if (slot_base >= 0) {
        for (int ai = 0; ai < na; ++ai) {
          uint32_t ov[8], rv[8];
          tc::ld8(tl + kTmO + 8 * ai, ov);
          tc::ld8(tl + kTmR + 8 * ai, rv);
          tc::wait_ld();
          const int64_t rec0 = ((int64_t)(slot_base + ai) * a.hkv + h) * G;
          const int r = row - kRank * ai;  // rank held by this lane of agent ai's rows of R
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < G) {
              a.part[(rec0 + q) * kPartCols + row] = nb > 0 ? __uint_as_float(ov[q]) : 0.f;
              if (r >= 0 && r < kRank) a.part[(rec0 + q) * kPartCols + kHeadDim + r] = nb > 0 ? __uint_as_float(rv[q]) : 0.f;
              if (row == kRank * na) {  // first row of the ones product: l
                a.ml[(rec0 + q) * 2] = nb > 0 && mref[ai * 8 + q] != kNoMax ? mref[ai * 8 + q] : -INFINITY;
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
  const int32_t* items;      // plan mode: the plan's work items (FORKKV_PLAN_ITEM_INTS each), else null
  int32_t n_items;
  const int32_t* seq_lens;   // [A]
  int32_t max_seq_len;
};

constexpr int kCombineChunk = 16;  // slots merged per pass (their partials held in registers)

// One CTA per (agent, KV head), one thread per (query head, d): log-sum-exp merge of the
// agent's partials, then out = (acc + acc_r B_v[:, hD:(h+1)D]) / l.  A pass brings the slot
// ids, then every (m, l) and this thread's partial of each slot at once, so that only three
// rounds of loads stand between the launch and the result; the running maximum carries
// across passes.
__global__ void __launch_bounds__(kMaxGroupQ * kHeadDim) decode_combine_kernel(const __grid_constant__ CombineArgs a) {
  const int agent = blockIdx.x, h = blockIdx.y, G = a.G;
  const int tid = threadIdx.x, gq = tid / kHeadDim, d = tid % kHeadDim;
  __shared__ int32_t s_slot[kCombineChunk];
  __shared__ float s_m[kMaxGroupQ][kCombineChunk], s_l[kMaxGroupQ][kCombineChunk];
  __shared__ float s_accr[kMaxGroupQ][kRank];
  __shared__ float s_lsum[kMaxGroupQ];
  __shared__ float s_bv[kRank][kHeadDim];  // B_v[:, hD:(h+1)D] of the agent's adapter
  int32_t s_begin, s_end;
  if (a.csr_off) {
    s_begin = a.csr_off[agent];
    s_end = a.csr_off[agent + 1];
  } else {
    s_begin = agent * a.chunks;
    s_end = s_begin + a.chunks;
  }
  if (s_begin < 0 || s_end < s_begin || s_end > a.n_slots) {
    if (tid == 0) flag_status(a.status, kDevBadArg);
    s_end = s_begin = 0;
  }
  if (a.items && h == 0) {
    // The plan's items of this agent must cover its pages exactly: a sequence that entered a new
    // page (or was truncated) after the plan was built would otherwise be attended partially.
    __shared__ int32_t s_pages;
    if (tid == 0) s_pages = 0;
    __syncthreads();
    int32_t pages = 0;
    for (int32_t i = tid; i < a.n_items; i += blockDim.x) {
      const int32_t* it = a.items + (int64_t)i * FORKKV_PLAN_ITEM_INTS;
      const int32_t na = it[2];
      bool mine = false;
      for (int x = 0; x < 8; ++x) mine |= x < na && it[4 + x] == agent;
      if (mine) pages += it[1] - it[0];
    }
    if (pages) atomicAdd(&s_pages, pages);
    __syncthreads();
    if (tid == 0 && s_pages != (min(a.seq_lens[agent], a.max_seq_len) + kPage - 1) / kPage)
      flag_status(a.status, kDevBadArg);
  }
  int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
  if ((uint32_t)adapter >= (uint32_t)a.n_adapters) adapter = 0;
  const __nv_bfloat16* Bv = a.B_v + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
  for (int i = tid; i < kRank * kHeadDim; i += blockDim.x)
    s_bv[i / kHeadDim][i % kHeadDim] = __bfloat162float(Bv[(int64_t)(i / kHeadDim) * a.hkv * kHeadDim + i % kHeadDim]);

  float M = -INFINITY, acc = 0.f, accr = 0.f, lsum = 0.f;
  for (int b0 = s_begin; b0 < s_end; b0 += kCombineChunk) {
    const int nb = min(kCombineChunk, s_end - b0);
    __syncthreads();  // the previous pass is done with the shared arrays
    if (tid < nb) {
      int32_t slot = a.csr_off ? a.csr_slots[b0 + tid] : b0 + tid;
      if ((uint32_t)slot >= (uint32_t)a.n_slots) {
        flag_status(a.status, kDevBadArg);
        slot = -1;
      }
      s_slot[tid] = slot;
    }
    __syncthreads();
    for (int i = tid; i < nb * G; i += blockDim.x) {  // (m, l) of every (slot, query head) of the pass
      const int gi = i / nb, si = i - gi * nb, slot = s_slot[si];
      const int64_t rec = ((int64_t)max(slot, 0) * a.hkv + h) * G + gi;
      s_m[gi][si] = slot >= 0 ? a.ml[rec * 2] : -INFINITY;
      s_l[gi][si] = slot >= 0 ? a.ml[rec * 2 + 1] : 0.f;
    }
    float pv[kCombineChunk], pr[kCombineChunk];  // this thread's partials of the pass
#pragma unroll
    for (int i = 0; i < kCombineChunk; ++i) {
      pv[i] = pr[i] = 0.f;
      if (i < nb) {
        const int64_t rec = ((int64_t)max(s_slot[i], 0) * a.hkv + h) * G + gq;
        pv[i] = a.part[rec * kPartCols + d];
        if (d < kRank) pr[i] = a.part[rec * kPartCols + kHeadDim + d];
      }
    }
    __syncthreads();
    float Mn = M;
    for (int i = 0; i < nb; ++i) Mn = fmaxf(Mn, s_m[gq][i]);
    if (Mn != -INFINITY) {
      const float sc = M == -INFINITY ? 0.f : exp2f(M - Mn);  // rescale what earlier passes gathered
      acc *= sc;
      accr *= sc;
      lsum *= sc;
#pragma unroll
      for (int i = 0; i < kCombineChunk; ++i)
        if (i < nb) {
          const float m = s_m[gq][i];
          const float w = m == -INFINITY ? 0.f : exp2f(m - Mn);
          acc += w * pv[i];
          accr += w * pr[i];
          lsum += w * s_l[gq][i];
        }
      M = Mn;
    }
  }
  if (d < kRank) s_accr[gq][d] = accr;
  if (d == 0) s_lsum[gq] = lsum;
  __syncthreads();
  float o = acc;
#pragma unroll
  for (int k = 0; k < kRank; ++k) o += s_accr[gq][k] * s_bv[k][d];
  lsum = s_lsum[gq];
  o = lsum > 0.f ? o / lsum : 0.f;
  a.out[((int64_t)agent * a.hkv * G + (int64_t)h * G + gq) * kHeadDim + d] = __float2bfloat16_rn(o);
}

}  // namespace

// SMs of the current device (the persistent decode grid is at most one CTA per SM); 152, a GB300,
// if the device does not answer.
static int32_t current_sm_count() {
  static thread_local int cached_dev = -1, cached_sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 152;
  }
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = 152;
    }
    cached_dev = dev;
    cached_sms = n;
  }
  return cached_sms;
}

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
    const int64_t want = current_sm_count();  // one CTA per SM
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
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sm_count = current_sm_count();
  if (configured_device != dev) {
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
  a.holes = p.holes;
  a.B_k = static_cast<const __nv_bfloat16*>(p.B_k);
  a.adapter_ids = p.adapter_ids;
  a.n_adapters = p.n_adapters;
  a.rope = static_cast<const uint8_t*>(rope_table);
  // whole pages of the table only (a page-major table holds positions in blocks of 16)
  a.rope_positions = p.rope_table ? p.rope_table_positions / kPage * kPage : (p.max_seq_len + kPage - 1) / kPage * kPage;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.0f / sqrtf((float)kHeadDim);
  a.scale_log2 = scale * 1.4426950408889634f;
  int32_t n_ctas;
  if (p.plan) {  // the unit records follow the items and the per-agent slot lists
    a.units = p.plan + (int64_t)p.plan_items * FORKKV_PLAN_ITEM_INTS + p.n_agents + 1 + p.plan_slots;
    a.n_units = p.plan_items * p.num_kv_heads;
    n_ctas = p.plan_ctas;
  } else {  // every (item, head) pair, dealt round-robin over at most one CTA per SM
    a.units = nullptr;
    a.n_units = g.n_items * p.num_kv_heads;
    n_ctas = (int32_t)std::min<int64_t>(a.n_units, std::max(1, sm_count));
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
    decode_split_kernel<4><<<n_ctas, kThreads, kSmemBytes, stream>>>(a);
  else
    decode_split_kernel<8><<<n_ctas, kThreads, kSmemBytes, stream>>>(a);
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
  c.items = p.plan;  // the items come first in a plan
  c.n_items = p.plan ? p.plan_items : 0;
  c.seq_lens = p.seq_lens;
  c.max_seq_len = p.max_seq_len;
  decode_combine_kernel<<<dim3(p.n_agents, p.num_kv_heads), G * kHeadDim, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace fkv
