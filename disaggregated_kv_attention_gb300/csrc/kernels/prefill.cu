// ResidualAttention over a prefill chunk for sm_103a, on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Same mathematics as decode (ForkKV L2 sections 4 and 7: deferred RoPE on the
// up-projected residual keys, associativity of the value path, both
// accumulators rescaled together), laid out for a dense contraction:
//   grid   (tile of 128 (token, query-head) rows, agent, KV head)
//   warps  0      producer: 128-key blocks (8 pages) of K and k_res tiles into a
//                 2-stage ring, V and v_res tiles into a 3-stage ring.  V and v_res
//                 go in as 1-D bulk async copies of one page tile each (several small
//                 copies land sooner than one large one).  K goes in as its two
//                 64-column halves, so that a stage holds the block's 128 keys as one
//                 K-major operand: when the block's 8 base pages are consecutive, one
//                 4-D tensor copy per half (8 pages of 16 rows), else one bulk copy per
//                 page half
//          1      allocates 512 TMEM columns; one lane issues every MMA
//          2..9   RoPE group, two warps per key (half of the rotation pairs each):
//                 U = Kr . B_k^T arrives in TMEM; K = bf16(Kb + RoPE_j(U)) replaces
//                 Kb in place in the stage, which the score MMA then reads
//          10..17 softmax group, two warps per query row (half of the keys each):
//                 S from TMEM, causal mask, online softmax; P (bf16) back into the
//                 block's TMEM buffer, over the S it came from, as the A operand of
//                 the value products
//   MMAs per block:  U[128x128]   = Kr[128x16] . B_k^T           (smem x smem)
//                    S[128x128]   = Q[128x128] . K^T             (smem x smem)
//                    O[128x128]  += P[128x128] . Vb[128x128]      (tmem x smem)
//                    O_r[128x16] += P . Vr[128x16]                (tmem x smem)
//   U, S and P of a block share one of two TMEM buffers (by block parity); U of
//   block b + 2 goes into the buffer once the value products of block b (the
//   last readers of its P) are done.  The next blocks' U, rotation and S run while this
//   block's softmax does; a K stage (a ring of three) is released by the commit
//   of its score MMA, so the rotation of block b + 1 overlaps the score product
//   of block b.  The MMA warp issues whichever product is ready first.
//   epilogue: out = (O + O_r . B_v[:, hD:(h+1)D]) / l, B_v applied once per row.
// Every wait is on an mbarrier with a bounded spin; a timeout sets the device
// status word instead of hanging.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "../internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fkv {
namespace {

constexpr int kRows = 128;
constexpr int kBlockPages = 8;
constexpr int kBlockKeys = kBlockPages * kPage;
constexpr int kRopeWarps = 8, kSoftWarp0 = 2 + kRopeWarps;  // warps 2..9 rotate keys, 10..17 run the softmax
constexpr int kThreads = (kSoftWarp0 + 8) * 32;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffPmax = 1024;                  // [2 parities][2 halves][128 rows] partial row maxima
constexpr int kKStages = 3, kVStages = 3;  // ring depths (at most 3 each)
// K stages: [the block's keys, K-major 128B-swizzled [2 halves][128 rows][128 B] | 8 k_res tiles];
// key 16 p + t of the block is row t of its page p, so half hh of page p's tile lands at
// hh * 16384 + p * 2048 and the swizzle (on row % 8 == t % 8) carries over unchanged
constexpr int kOffKStage = 3072;
constexpr int kOffVStage = kOffKStage + kKStages * 36864;  // V stages of [8 V tiles | 8 v_res tiles]
constexpr int kStageBytes = 36864, kStRes = 32768;  // the residual tiles follow the base tiles
constexpr int kOffBk = kOffVStage + kVStages * kStageBytes;  // B_k^T, K-major 32B-swizzled [128 d][16 r]
constexpr int kOffBv = kOffBk + 4096;                         // B_v slice [16][128] bf16
constexpr int kSmemBytes = kOffBv + 4096;  // the dynamic window is 1024-byte aligned (checked)
static_assert(kSmemBytes <= 227 * 1024, "more shared memory than a CTA may have");

// tensor memory columns: two buffers (U, then S, then P over S) by block parity, O, O_r
// and Q (bf16 pairs: the A operand of the score product).  P of the keys 64 sh .. 64 sh + 63
// (bf16 pairs) sits at columns 64 sh .. 64 sh + 31 of its buffer, under the S columns that the
// softmax warps of half sh themselves read.
constexpr uint32_t kTmBuf = 0, kTmO = 256, kTmOr = 384, kTmQ = 400, kTmCols = 512;

// mbarrier indices
enum { kKFull0, kKFull1, kKFull2, kKEmpty0, kKEmpty1, kKEmpty2, kVFull0, kVFull1, kVFull2, kVEmpty0, kVEmpty1, kVEmpty2,
       kUFull0, kUFull1,
       kKFReady0, kKFReady1, kKFReady2, kSFull0, kSFull1,
       kPFull0, kPFull1, kPVDone0, kPVDone1, kQReady, kBkReady, kMmaDone, kNumBars };
static_assert(kNumBars * 8 <= 256, "barriers overlap the state that follows them");

// Bytes of nvp page tiles whose last page keeps only `rows` rows.
__device__ __forceinline__ uint32_t tile_bytes_pf(bool base, int nvp, int rows) {
  const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
  return rows < kPage ? (uint32_t)(nvp - 1) * tile + (base ? 2u : 1u) * (uint32_t)rows * rb : (uint32_t)nvp * tile;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 values in one 64-bit register for the packed fp32 instructions (add/fma .f32x2);
// each lane rounds exactly as the scalar instruction does.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}


struct PrefillArgs {
  // This layer's base K pool as [Hkv * pages][2 halves][16 rows][128 B]: a box of 8 pages of one
  // half lands in shared memory as the rows of 128 keys of one 64-column block.
  CUtensorMap kb_map;
  int32_t kb_map_ok;
  const uint8_t* k_base;
  const uint8_t* v_base;
  const uint8_t* k_res;
  const uint8_t* v_res;
  int32_t num_base_pages, num_res_pages, hkv, G, q_len, n_agents;
  const __nv_bfloat16* q;  // [A][q_len][Hq][128]
  __nv_bfloat16* out;
  const int32_t* bpt;
  const int32_t* rpt;
  int32_t pt_stride, max_seq_len;
  const int32_t* seq_lens;
  const int32_t* positions;  // [A][q_len]
  const int32_t* holes;      // [A][2] slot map (first hole slot, hole length), or null
  const __nv_bfloat16* B_k;
  const __nv_bfloat16* B_v;
  const int32_t* adapter_ids;
  int32_t n_adapters;
  const uint8_t* rope;
  int32_t rope_positions;
  float scale_log2;
  uint32_t* status;
};


__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023) {  // swizzled operand tiles need a 1024-byte aligned window
    if (threadIdx.x == 0) flag_status(a.status, kDevBadArg);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + 256);
  int32_t* s_meta = reinterpret_cast<int32_t*>(smem + 272);
  float* s_pmax = reinterpret_cast<float*>(smem + kOffPmax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int agent = blockIdx.y, h = blockIdx.z;
  const int G = a.G;
  const int64_t n_rows = (int64_t)a.q_len * G;
  const int64_t row0 = (int64_t)blockIdx.x * kRows;
  const int32_t L = min(a.seq_lens[agent], a.max_seq_len);
  int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
  if ((uint32_t)adapter >= (uint32_t)a.n_adapters) adapter = 0;
  // the agent's slot map: the key in slot j is hidden in [hs, hs + hn) and sits at position
  // j - hn past it (kpos); token position p sits in slot p, or p + hn from hs on
  int32_t hs = a.holes ? a.holes[2 * agent] : 0, hn = a.holes ? a.holes[2 * agent + 1] : 0;
  if (hn < 0 || hn >= kPage || hs < 0) {
    if (threadIdx.x == 0) flag_status(a.status, kDevBadArg);
    hs = hn = 0;
  }
  auto kpos = [&](int j) { return (hn != 0 && j >= hs + hn) ? j - hn : j; };
  // key positions grow with the slot, so "position <= p" is "slot <= slot of p" (hole aside)
  auto slot_of = [&](int32_t p) { return (hn != 0 && p >= hs) ? p + hn : p; };
  const int32_t hlo = hn != 0 ? hs : 0, hhi = hn != 0 ? hs + hn : 0;  // hidden slots [hlo, hhi)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars[kKFull0 + i], 1);
      mbar_init(&bars[kKEmpty0 + i], 1);            // the commit after the score MMA
      mbar_init(&bars[kKFReady0 + i], kRopeWarps);  // every RoPE warp, once its keys are rotated
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars[kVFull0 + i], 1);
      mbar_init(&bars[kVEmpty0 + i], 1);  // the commit after the value products
    }
    mbar_init(&bars[kUFull0], 1);
    mbar_init(&bars[kUFull1], 1);
    mbar_init(&bars[kSFull0], 1);
    mbar_init(&bars[kSFull1], 1);
    // P written, by block parity: a softmax warp may write P of block b + 1 before a slower one
    // has written P of block b, and on a single barrier its arrival would complete block b's
    // phase early; it cannot reach block b + 2 before block b's value products are done
    mbar_init(&bars[kPFull0], 8);  // every softmax warp
    mbar_init(&bars[kPFull1], 8);
    mbar_init(&bars[kPVDone0], 1);  // the commit after the value products of an even block
    mbar_init(&bars[kPVDone1], 1);  // of an odd block
    mbar_init(&bars[kQReady], 8);
    mbar_init(&bars[kBkReady], kRopeWarps);
    mbar_init(&bars[kMmaDone], 1);
    mbar_fence_init();
    // keys this CTA may see: up to the largest query position of its rows (and L)
    const int t_first = (int)(row0 / G);
    const int t_last = (int)((min(row0 + kRows, n_rows) - 1) / G);
    int32_t pmax = -1;
    bool bad_pos = false;  // a query position must name a slot of the sequence: 0 <= p, slot_of(p) < seq_len
    for (int t = t_first; t <= t_last; ++t) {
      const int32_t pt = a.positions[(int64_t)agent * a.q_len + t];
      bad_pos |= pt < 0 || slot_of(pt) >= a.seq_lens[agent];
      pmax = max(pmax, pt);
    }
    if (bad_pos) flag_status(a.status, kDevBadArg);
    if (a.seq_lens[agent] < 1 || a.seq_lens[agent] > a.max_seq_len) flag_status(a.status, kDevBadArg);
    if ((uint32_t)(a.adapter_ids ? a.adapter_ids[agent] : agent) >= (uint32_t)a.n_adapters)
      flag_status(a.status, kDevBadArg);
    s_meta[0] = max(0, min(slot_of(pmax) + 1, L));
  }
  if (warp == 1) tc::alloc(s_tmem, kTmCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = *s_tmem;
  const int32_t key_limit = s_meta[0];
  const int n_pages = (key_limit + kPage - 1) / kPage;
  const int n_blocks = (n_pages + kBlockPages - 1) / kBlockPages;
  uint8_t* sBk = smem + kOffBk;
  uint8_t* sBv = smem + kOffBv;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    // Two streams in block order, K ahead of V: a block's K and k_res tiles once the score
    // product of the block kKStages back is done with that K stage, its V and v_res tiles once
    // the value products of the block kVStages back are done with that V stage.  Rows of the
    // last page at or past the sequence end are zeroed in shared memory instead of copied, so that
    // a zero probability never meets never-written (possibly NaN) value rows.
    const int64_t head_base = (int64_t)h * a.num_base_pages;
    // page id of block b held by this lane (lanes 0..7 the base pages, 8..15 the residual
    // pages; requested, not waited for)
    auto lane_id = [&](int b) -> int32_t {
      const int pbase = b * kBlockPages, nvp = min(kBlockPages, n_pages - pbase);
      int32_t id = 0;
      if (lane < nvp) id = a.bpt[(int64_t)agent * a.pt_stride + pbase + lane];
      else if (lane >= 8 && lane - 8 < nvp) id = a.rpt[(int64_t)agent * a.pt_stride + pbase + lane - 8];
      return id;
    };
    // the ids of a block to its copying lanes: lane 0 the base ids, lanes 1 and 16 the residual ids
    auto broadcast_ids = [&](int b, int32_t& id, int32_t (&ids)[8]) {
      const int nvp = min(kBlockPages, n_pages - b * kBlockPages);
      if (lane < nvp && (uint32_t)id >= (uint32_t)a.num_base_pages) {
        flag_status(a.status, kDevBadPage);
        id = 0;
      } else if (lane >= 8 && lane - 8 < nvp && (uint32_t)id >= (uint32_t)a.num_res_pages) {
        flag_status(a.status, kDevBadPage);
        id = 0;
      }
      const int src0 = (lane == 1 || lane == 16) ? 8 : 0;
#pragma unroll
      for (int pg = 0; pg < 8; ++pg) ids[pg] = __shfl_sync(0xffffffffu, id, src0 + pg);
    };
    // one lane's copies of a block: whole pages by runs of consecutive ids, then the first
    // `rows` rows of the last page when rows < 16
    auto copy_pages = [&](const uint8_t* pool, uint8_t* dst, bool base, const int32_t (&ids)[8], int nvp, int rows,
                          uint64_t* bar) {
      const uint32_t tile = base ? kBaseTile : kResTile, rb = base ? 128u : 32u;
      const int full = rows < kPage ? nvp - 1 : nvp;
      int r0 = 0;
      int32_t start = ids[0];
#pragma unroll
      for (int pg = 1; pg <= 8; ++pg) {
        if (pg <= full) {
          const bool end = pg == full || ids[pg < 8 ? pg : 7] != ids[pg - 1] + 1;
          if (end) {
            bulk_g2s(dst + r0 * tile, pool + (int64_t)start * tile, (pg - r0) * tile, bar);
            r0 = pg;
            start = ids[pg < 8 ? pg : 7];
          }
        }
      }
      if (full < nvp && rows > 0) {
        int32_t id = ids[0];
#pragma unroll
        for (int pg = 1; pg < 8; ++pg)
          if (pg == full) id = ids[pg];
        const uint8_t* src = pool + (int64_t)id * tile;
        bulk_g2s(dst + full * tile, src, rows * rb, bar);
        if (base) bulk_g2s(dst + full * tile + 2048, src + 2048, rows * rb, bar);
      }
    };
    // K copies of block b (ids in idsb; `id` this lane's checked id), once its stage is free:
    // lane 2 p + hh copies half hh of page p's K tile, lane 16 the k_res tiles
    auto copy_k = [&](int b, const int32_t (&idsb)[8], int32_t id) {
      const int stage = b % kKStages;
      const int nvp = min(kBlockPages, n_pages - b * kBlockPages);
      uint8_t* st = smem + kOffKStage + stage * kStageBytes;
      const int32_t pid = __shfl_sync(0xffffffffu, id, (lane >> 1) & 7);
      if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull0 + stage], nvp * (kBaseTile + kResTile));
      __syncwarp();
      // eight consecutive base pages: one tensor copy per 64-column half instead of 16 page halves
      const int32_t pid0 = __shfl_sync(0xffffffffu, id, 0);
      const bool run = a.kb_map_ok && nvp == kBlockPages &&
                       __all_sync(0xffffffffu, lane >= 16 || pid == pid0 + ((lane >> 1) & 7));
      if (run) {
        if (lane < 2) tma_load_kb(st + lane * 16384, &a.kb_map, lane, (int32_t)(head_base + pid0), &bars[kKFull0 + stage]);
      } else if (lane < 2 * nvp) {
        const int hh = lane & 1;
        bulk_g2s(st + hh * 16384 + (lane >> 1) * 2048, a.k_base + (head_base + pid) * kBaseTile + hh * 2048,
                 kBaseTile / 2, &bars[kKFull0 + stage]);
      }
      if (lane == 16) copy_pages(a.k_res, st + kStRes, false, idsb, nvp, kPage, &bars[kKFull0 + stage]);
    };
    // V copies of block b (`id` this lane's checked id), once its V stage is free
    auto copy_v = [&](int b, int32_t id) {
      const int nvp = min(kBlockPages, n_pages - b * kBlockPages);
      const int rows = b * kBlockPages + nvp == n_pages ? min(kPage, max(0, L - (n_pages - 1) * kPage)) : kPage;
      uint8_t* st = smem + kOffVStage + (b % kVStages) * kStageBytes;
      uint64_t* vbar = &bars[kVFull0 + b % kVStages];
      if (rows < kPage) {  // rows [rows, 16) of the last V and v_res tiles
        uint8_t* tv = st + (nvp - 1) * kBaseTile;
        uint8_t* tr = st + kStRes + (nvp - 1) * kResTile;
        for (int o = rows * 128 + 16 * lane; o < 2048; o += 16 * 32) {
          *reinterpret_cast<uint4*>(tv + o) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(tv + 2048 + o) = make_uint4(0u, 0u, 0u, 0u);
        }
        for (int o = rows * 32 + 16 * lane; o < kResTile; o += 16 * 32)
          *reinterpret_cast<uint4*>(tr + o) = make_uint4(0u, 0u, 0u, 0u);
        tc::fence_proxy_async();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(vbar, tile_bytes_pf(true, nvp, rows) + tile_bytes_pf(false, nvp, rows));
      __syncwarp();
      // one copy per page tile: lane pg the V tile of page pg, lane 8 + pg its v_res tile (the
      // first `rows` rows of each half for the last page when rows < 16)
      const int pg = lane & 7;
      const int32_t pid = __shfl_sync(0xffffffffu, id, lane & 15);
      const bool last = pg == nvp - 1 && rows < kPage;
      if (lane < 8 && pg < nvp) {
        const uint8_t* src = a.v_base + (head_base + pid) * kBaseTile;
        if (!last) {
          bulk_g2s(st + pg * kBaseTile, src, kBaseTile, vbar);
        } else if (rows > 0) {
          bulk_g2s(st + pg * kBaseTile, src, rows * 128, vbar);
          bulk_g2s(st + pg * kBaseTile + 2048, src + 2048, rows * 128, vbar);
        }
      } else if (lane >= 8 && lane < 16 && pg < nvp && (!last || rows > 0)) {
        bulk_g2s(st + kStRes + pg * kResTile, a.v_res + (int64_t)pid * kResTile, last ? rows * 32 : kResTile, vbar);
      }
    };
    // Two streams without waiting on each other (K ahead of V as far as its stages allow).  Each
    // stream holds this lane's page ids of its next three blocks (kq0..2, vq0..2): an id load
    // takes microseconds while every SM streams, so it is requested three copies ahead.
    int32_t ids[8];
    int32_t kq0 = lane_id(0), kq1 = lane_id(1), kq2 = lane_id(2);
    int32_t vq0 = kq0, vq1 = kq1, vq2 = kq2;
    int kb = 0, vb = 0;  // next K block, next V block
    uint32_t idle = 0;
    bool ok = true;
    while (ok && vb < n_blocks) {
      bool did = false;
      if (kb < n_blocks &&
          __shfl_sync(0xffffffffu, kb < kKStages || mbar_test(&bars[kKEmpty0 + kb % kKStages], (kb / kKStages - 1) & 1),
                      0)) {
        broadcast_ids(kb, kq0, ids);
        copy_k(kb, ids, kq0);
        ++kb;
        kq0 = kq1;
        kq1 = kq2;
        kq2 = lane_id(kb + 2);  // 0 past the last block
        did = true;
      }
      if (vb < kb &&
          __shfl_sync(0xffffffffu, vb < kVStages || mbar_test(&bars[kVEmpty0 + vb % kVStages], (vb / kVStages - 1) & 1),
                      0)) {
        broadcast_ids(vb, vq0, ids);
        copy_v(vb, vq0);
        ++vb;
        vq0 = vq1;
        vq1 = vq2;
        vq2 = lane_id(vb + 2);
        did = true;
      }
      if (did) {
        idle = 0;
      } else {
        if (++idle > kWaitLimit) {
          flag_status(a.status, kDevTimeout);
          ok = false;
        }
        __nanosleep(100);
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // Issues, whichever is ready first (scores first: the softmax waits on them and the value
    // products of the previous block need only be done before the next P is written; then the
    // value products, then U):
    //   U(b)  into buffer b % 2 once block b's K stage is in and P.V(b - 2), the last reader of
    //         that buffer, is done;
    //   S(b)  over U(b) once the rotation group has built K(b) in its stage (whose commit then
    //         frees the stage for block b + 3);
    //   P.V(b) once the softmax has written P(b) and block b's V stage is in.
    if (lane == 0) {
      const uint32_t idU = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idS = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idPV = tc::idesc_bf16(128, 128, 0, 1);
      const uint32_t idPVr = tc::idesc_bf16(128, 16, 0, 1);
      const uint32_t aK = smem_u32(smem + kOffKStage), aBk = smem_u32(sBk);
      bool ok = mbar_wait(&bars[kQReady], 0, a.status) && mbar_wait(&bars[kBkReady], 0, a.status);
      int iu = 0, is = 0, ip = 0;  // next U, S and P.V to issue
      uint32_t idle = 0;
      while (ok && ip < n_blocks) {
        bool did = false;
        if (is < iu && mbar_test(&bars[kKFReady0 + is % kKStages], (is / kKStages) & 1)) {
          tc::fence_after();
          const uint32_t buf = tm + kTmBuf + 128 * (is & 1);
          const uint32_t aKs = aK + (is % kKStages) * kStageBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
            tc::mma_ts(buf, tm + kTmQ + 8 * ks, tc::smem_desc(aKs + off, 16, 1024, tc::kSwizzle128B), idS, ks > 0);
          }
          tc::commit(&bars[kSFull0 + (is & 1)]);
          tc::commit(&bars[kKEmpty0 + is % kKStages]);
          ++is;
          did = true;
        }
        if (ip < is && mbar_test(&bars[kPFull0 + (ip & 1)], (ip >> 1) & 1) &&
            mbar_test(&bars[kVFull0 + ip % kVStages], (ip / kVStages) & 1)) {
          tc::fence_after();
          const uint32_t aV = smem_u32(smem + kOffVStage + (ip % kVStages) * kStageBytes);
          const int nvp = min(kBlockPages, n_pages - ip * kBlockPages);
          // P of keys 16 ks .. 16 ks + 15: 8 columns of the block's buffer (keys 64 .. at column 64)
          const uint32_t pb = tm + kTmBuf + 128 * (ip & 1);
          for (int ks = 0; ks < nvp; ++ks)  // 16 keys per step: one V tile
            tc::mma_ts(tm + kTmO, pb + (ks >> 2) * 64 + (ks & 3) * 8,
                       tc::smem_desc(aV + ks * kBaseTile, 2048, 1024, tc::kSwizzle128B), idPV, (ip > 0 || ks > 0));
          for (int ks = 0; ks < nvp; ++ks)
            tc::mma_ts(tm + kTmOr, pb + (ks >> 2) * 64 + (ks & 3) * 8,
                       tc::smem_desc(aV + kStRes + ks * kResTile, 4096, 256, tc::kSwizzle32B), idPVr, (ip > 0 || ks > 0));
          tc::commit(&bars[kPVDone0 + (ip & 1)]);
          tc::commit(&bars[kVEmpty0 + ip % kVStages]);
          ++ip;
          did = true;
        }
        if (iu < n_blocks && iu - is < 2 && mbar_test(&bars[kKFull0 + iu % kKStages], (iu / kKStages) & 1) &&
            (iu < 2 || (ip + 2 > iu && mbar_test(&bars[kPVDone0 + (iu & 1)], ((iu >> 1) - 1) & 1)))) {
          tc::fence_after();
          const uint32_t st = aK + (iu % kKStages) * kStageBytes;
          tc::mma_ss(tm + kTmBuf + 128 * (iu & 1), tc::smem_desc(st + kStRes, 16, 256, tc::kSwizzle32B),
                     tc::smem_desc(aBk, 16, 256, tc::kSwizzle32B), idU, 0);
          tc::commit(&bars[kUFull0 + (iu & 1)]);
          ++iu;
          did = true;
        }
        if (did) {
          idle = 0;
        } else {
          if (++idle > kWaitLimit) {
            flag_status(a.status, kDevTimeout);
            ok = false;
          }
          // sleep on the event due first
          if (ip < is)
            mbar_try_wait_for(&bars[kPFull0 + (ip & 1)], (ip >> 1) & 1, 200);
          else if (is < iu)
            mbar_try_wait_for(&bars[kKFReady0 + is % kKStages], (is / kKStages) & 1, 200);
          else
            mbar_try_wait_for(&bars[kKFull0 + iu % kKStages], (iu / kKStages) & 1, 200);
        }
      }
      // never leave with MMAs in flight
      tc::commit(&bars[kMmaDone]);
      mbar_wait(&bars[kMmaDone], 0, a.status);
    }
    __syncwarp();
  } else if (warp < kSoftWarp0) {
    // ------------------------------ RoPE group ------------------------------
    // Two warps per TMEM lane quadrant; half hf owns the rotation pairs (d, d + 64) with
    // d in [32 hf, 32 hf + 32) of its 32 keys.
    const int hf = (warp - 2) >> 2;
    const int row = 32 * (warp & 3) + lane;  // key row of the block == TMEM lane
    const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    {  // B_k^T: row d, this half's 8 of the 16 ranks
      const __nv_bfloat16* B = a.B_k + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim + row;
#pragma unroll
      for (int k = 8 * hf; k < 8 * hf + 8; ++k)
        *reinterpret_cast<__nv_bfloat16*>(sBk + tc::sw32_off(row, k)) = B[(int64_t)k * a.hkv * kHeadDim];
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBkReady]);
    }
    bool ok = true;
    for (int b = 0; b < n_blocks && ok; ++b) {
      const int stage = b % kKStages;
      uint8_t* st = smem + kOffKStage + stage * kStageBytes;
      const uint32_t ub = tl + kTmBuf + 128 * (b & 1);
      const int j = b * kBlockKeys + row;
      const int jr = kpos(j) < a.rope_positions ? kpos(j) : 0;
      // this key's rotation entries (position jr): frequency groups 4 u .. 4 u + 3 are 32 bytes
      // at rope_off(jr, 4 u); this half needs u = 4 hf .. 4 hf + 3
      const uint8_t* rrow = a.rope + rope_off(jr, 0);
      uint4 rp[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        rp[u][0] = *reinterpret_cast<const uint4*>(rrow + (4 * hf + u) * 512);
        rp[u][1] = *reinterpret_cast<const uint4*>(rrow + (4 * hf + u) * 512 + 16);
      }
      ok = mbar_wait(&bars[kKFull0 + stage], (b / kKStages) & 1, a.status) &&
           mbar_wait(&bars[kUFull0 + (b & 1)], (b >> 1) & 1, a.status);
      if (!ok) break;
      tc::fence_after();
#pragma unroll
      for (int c = 32 * hf; c < 32 * hf + 32; c += 16) {  // d in [c, c + 16) and [c + 64, c + 80)
        uint32_t ulo[16], uhi[16];
        tc::ld16(ub + c, ulo);
        tc::ld16(ub + 64 + c, uhi);
        uint4 kl[2], kh[2];
        kl[0] = *reinterpret_cast<const uint4*>(st + tc::sw128_off(128, row, c));
        kl[1] = *reinterpret_cast<const uint4*>(st + tc::sw128_off(128, row, c + 8));
        kh[0] = *reinterpret_cast<const uint4*>(st + tc::sw128_off(128, row, c + 64));
        kh[1] = *reinterpret_cast<const uint4*>(st + tc::sw128_off(128, row, c + 72));
        tc::wait_ld();
        const uint32_t* klw = reinterpret_cast<const uint32_t*>(kl);
        const uint32_t* khw = reinterpret_cast<const uint32_t*>(kh);
        uint32_t olo[8], ohi[8];
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {  // frequency group c/2 + i2: elements d = c + 2 i2, + 1 (and + 64)
          const int m = ((c - 32 * hf) >> 1) + i2;  // frequency group, counted from 16 hf
          const uint4 w = rp[m >> 2][(m & 3) >> 1];
          const uint32_t cw = (m & 1) ? w.z : w.x, sw = (m & 1) ? w.w : w.y;
          // K = Kb + RoPE_j(U) in fp32, one bf16 rounding
          const float lo0 = __uint_as_float(ulo[2 * i2]), lo1 = __uint_as_float(ulo[2 * i2 + 1]);
          const float hi0 = __uint_as_float(uhi[2 * i2]), hi1 = __uint_as_float(uhi[2 * i2 + 1]);
          const float c0 = bf_lo(cw), c1 = bf_hi(cw), s0 = bf_lo(sw), s1 = bf_hi(sw);
          olo[i2] = pack_bf16(fmaf(lo0, c0, fmaf(-hi0, s0, bf_lo(klw[i2]))), fmaf(lo1, c1, fmaf(-hi1, s1, bf_hi(klw[i2]))));
          ohi[i2] = pack_bf16(fmaf(hi0, c0, fmaf(lo0, s0, bf_lo(khw[i2]))), fmaf(hi1, c1, fmaf(lo1, s1, bf_hi(khw[i2]))));
        }
        // in place: this thread alone reads and writes these elements of its key row
        *reinterpret_cast<uint4*>(st + tc::sw128_off(128, row, c)) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
        *reinterpret_cast<uint4*>(st + tc::sw128_off(128, row, c + 8)) = make_uint4(olo[4], olo[5], olo[6], olo[7]);
        *reinterpret_cast<uint4*>(st + tc::sw128_off(128, row, c + 64)) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
        *reinterpret_cast<uint4*>(st + tc::sw128_off(128, row, c + 72)) = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      }
      tc::fence_before();
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kKFReady0 + stage]);
      }
    }
  } else {
    // ------------------------------ softmax group ------------------------------
    // Two warps per TMEM lane quadrant: half sh holds the keys [64 sh, 64 sh + 64) of each
    // block and the output columns d in [64 sh, 64 sh + 64); the two halves of a row meet
    // through shared memory and a named barrier (one per quadrant).
    const int q4 = warp & 3, sh = (warp - kSoftWarp0) >> 2;
    const int qr = 32 * q4 + lane;  // query row of the tile == TMEM lane
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);
    const uint32_t pair_bar = 1 + q4, pair_threads = 64;
    const int64_t f = row0 + qr;
    const bool valid = f < n_rows;
    const int64_t tq = valid ? f / G : 0;
    const int gq = valid ? (int)(f % G) : 0;
    const int32_t pos = valid ? a.positions[(int64_t)agent * a.q_len + tq] : -1;
    const int32_t lim = min(L, slot_of(pos) + 1);  // slots below lim (outside the hole) are visible
    const int64_t orow = (((int64_t)agent * a.q_len + tq) * a.hkv * G + (int64_t)h * G + gq) * kHeadDim;
    {  // this half of the Q row into tensor memory (d = 64 sh .. 64 sh + 63 as bf16 pairs in
       // columns 32 sh ..); this half of the B_v slice
      const uint4* src = reinterpret_cast<const uint4*>(a.q + orow);
      uint32_t qw[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 v = valid ? src[8 * sh + i] : make_uint4(0u, 0u, 0u, 0u);
        qw[4 * i] = v.x;
        qw[4 * i + 1] = v.y;
        qw[4 * i + 2] = v.z;
        qw[4 * i + 3] = v.w;
      }
      tc::st16(tl + kTmQ + 32 * sh, qw);
      tc::st16(tl + kTmQ + 32 * sh + 16, qw + 16);
      tc::wait_st();
      tc::fence_before();
      const __nv_bfloat16* Bv = a.B_v + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
      for (int i = qr + 128 * sh; i < kRank * kHeadDim / 8; i += 256) {
        const int k = i / 16, ch = i % 16;
        *reinterpret_cast<uint4*>(sBv + (k * kHeadDim + ch * 8) * 2) =
            *reinterpret_cast<const uint4*>(Bv + (int64_t)k * a.hkv * kHeadDim + ch * 8);
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kQReady]);
    }
    float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
    bool ok = true;
    // No early exit: both warps of a quadrant take every named barrier; after a wait that timed
    // out (the status word says so) the loop runs on without waiting and its values are void.
    for (int b = 0; b < n_blocks; ++b) {
      const uint32_t buf = kTmBuf + 128 * (b & 1);
      ok = ok && mbar_wait(&bars[kSFull0 + (b & 1)], (b >> 1) & 1, a.status);
      tc::fence_after();
      const int kbase = b * kBlockKeys + 64 * sh;
      // keys of this half all visible to this row: no per-key mask (every block below the diagonal)
      const bool open = kbase + 64 <= lim && !(kbase < hhi && kbase + 64 > hlo);
      float bm = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t v[32];
        tc::ld16(tl + buf + 64 * sh + c, v);
        tc::ld16(tl + buf + 64 * sh + c + 16, v + 16);
        tc::wait_ld();
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (open) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx[(i >> 1) & 3] = max3(mx[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int j = kbase + c + i;
            if (j < lim && (j < hlo || j >= hhi)) mx[i & 3] = fmaxf(mx[i & 3], __uint_as_float(v[i]));
          }
        }
        bm = fmaxf(bm, fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])));
      }
      bm *= a.scale_log2;  // the scale is positive, so it commutes with the maximum
      // the row's block maximum: both halves (parity-alternating slots, so one barrier per block)
      s_pmax[((b & 1) * 2 + sh) * 128 + qr] = bm;
      named_sync(pair_bar, pair_threads);
      bm = fmaxf(bm, s_pmax[((b & 1) * 2 + (sh ^ 1)) * 128 + qr]);
      const bool need = bm > m + 8.f;  // lazy rescale: only when the max grows by 2^8
      if (__any_sync(0xffffffffu, need)) {
        const float mn = need ? bm : m;
        const float alpha = (need && m != -INFINITY) ? exp2f(m - mn) : 1.f;
        if (b > 0) {
          // O (this half's columns; the first half also O_r) is stable once P.V of block b - 1 is done
          ok = ok && mbar_wait(&bars[kPVDone0 + ((b - 1) & 1)], ((b - 1) >> 1) & 1, a.status);
          tc::fence_after();
#pragma unroll
          for (int c = 0; c < 64 + 16; c += 16) {
            if (c == 64 && sh == 1) break;
            const uint32_t col = c < 64 ? kTmO + 64 * sh + c : kTmOr;
            uint32_t v[16];
            tc::ld16(tl + col, v);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tc::st16(tl + col, v);
          }
          tc::wait_st();
        }
        l *= alpha;
        m = mn;
      }
      const float mu = m == -INFINITY ? 0.f : m;
      // P of this half's keys (64 sh + 2 i, 2 i + 1 in pw[i]): p = 2^(s * scale - mu) in one
      // multiply-add, the row sum in four partial sums (two packed pairs)
      const uint64_t sc2 = f2(a.scale_log2, a.scale_log2), nmu2 = f2(-mu, -mu);
      uint64_t ls2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
      uint32_t pw[32];
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t v[32];
        tc::ld16(tl + buf + 64 * sh + c, v);
        tc::ld16(tl + buf + 64 * sh + c + 16, v + 16);
        tc::wait_ld();
        if (open) {  // every key of this half is visible to the row
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sc2, nmu2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            ls2[i & 1] = f2_add(ls2[i & 1], f2(p0, p1));
            pw[(c >> 1) + i] = pack_bf16(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float pr[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int j = kbase + c + 2 * i + e;
              const float x = ex2(fmaf(__uint_as_float(v[2 * i + e]), a.scale_log2, -mu));
              pr[e] = (j < lim && (j < hlo || j >= hhi)) ? x : 0.f;
            }
            ls2[i & 1] = f2_add(ls2[i & 1], f2(pr[0], pr[1]));
            pw[(c >> 1) + i] = pack_bf16(pr[0], pr[1]);
          }
        }
      }
      {
        float l0, l1, l2, l3;
        f2_split(ls2[0], l0, l1);
        f2_split(ls2[1], l2, l3);
        l += (l0 + l1) + (l2 + l3);
      }
      // P of this half's keys (bf16 pairs) into the block's buffer over the S columns this half
      // has read (the buffer's previous P, of block b - 2, was done with before U(b) went in)
      tc::st16(tl + buf + 64 * sh, pw);
      tc::st16(tl + buf + 64 * sh + 16, pw + 16);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kPFull0 + (b & 1)]);
    }
    // epilogue: the row sum of both halves, then this half's output columns
    if (ok && n_blocks > 0) ok = mbar_wait(&bars[kPVDone0 + ((n_blocks - 1) & 1)], ((n_blocks - 1) >> 1) & 1, a.status);
    if (ok) ok = mbar_wait(&bars[kQReady], 0, a.status);  // every thread's part of the B_v slice is in place
    named_sync(pair_bar, pair_threads);  // both halves are past their last use of s_pmax
    s_pmax[sh * 128 + qr] = l;
    named_sync(pair_bar, pair_threads);
    l += s_pmax[(sh ^ 1) * 128 + qr];
    tc::fence_after();
    uint32_t orr[16];
    tc::ld16(tl + kTmOr, orr);
    tc::wait_ld();
    const bool have = ok && n_blocks > 0 && l > 0.f;
    const float inv = have ? 1.f / l : 0.f;
    const __nv_bfloat16* sbv = reinterpret_cast<const __nv_bfloat16*>(sBv);
#pragma unroll 1
    for (int c = 64 * sh; c < 64 * sh + 64; c += 16) {
      uint32_t v[16];
      tc::ld16(tl + kTmO + c, v);
      tc::wait_ld();
      uint32_t ow[8];
#pragma unroll
      for (int i2 = 0; i2 < 8; ++i2) {
        float o[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = c + 2 * i2 + e;
          float x = __uint_as_float(v[2 * i2 + e]);
#pragma unroll
          for (int k = 0; k < kRank; ++k) x += __uint_as_float(orr[k]) * __bfloat162float(sbv[k * kHeadDim + d]);
          o[e] = have ? x * inv : 0.f;
        }
        ow[i2] = pack_bf16(o[0], o[1]);
      }
      if (valid) {
        uint4* dst = reinterpret_cast<uint4*>(a.out + orow + c);
        dst[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
        dst[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tm, kTmCols);
  }
}

}  // namespace

// cuTensorMapEncodeTiled through the runtime's driver entry point (nullptr if unavailable).
static PFN_cuTensorMapEncodeTiled_v12000 kb_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

cudaError_t launch_prefill(const forkkv_attn_params& p, const void* rope_table, uint32_t* status,
                           cudaStream_t stream) {
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const int32_t G = p.num_q_heads / p.num_kv_heads;
  const int64_t base_layer = (int64_t)p.pools.num_base_pages * p.pools.num_kv_heads * kBaseTile;
  const int64_t res_layer = (int64_t)p.pools.num_res_pages * kResTile;
  PrefillArgs a;
  a.k_base = static_cast<const uint8_t*>(p.pools.k_base) + p.layer * base_layer;
  a.v_base = static_cast<const uint8_t*>(p.pools.v_base) + p.layer * base_layer;
  a.k_res = static_cast<const uint8_t*>(p.pools.k_res) + p.layer * res_layer;
  a.v_res = static_cast<const uint8_t*>(p.pools.v_res) + p.layer * res_layer;
  a.num_base_pages = p.pools.num_base_pages;
  a.num_res_pages = p.pools.num_res_pages;
  a.hkv = p.num_kv_heads;
  a.G = G;
  a.q_len = p.q_len;
  a.n_agents = p.n_agents;
  a.q = static_cast<const __nv_bfloat16*>(p.q);
  a.out = static_cast<__nv_bfloat16*>(p.out);
  a.bpt = p.bpt;
  a.rpt = p.rpt;
  a.pt_stride = p.pt_stride;
  a.max_seq_len = p.max_seq_len;
  a.seq_lens = p.seq_lens;
  a.positions = p.positions;
  a.holes = p.holes;
  a.B_k = static_cast<const __nv_bfloat16*>(p.B_k);
  a.B_v = static_cast<const __nv_bfloat16*>(p.B_v);
  a.adapter_ids = p.adapter_ids;
  a.n_adapters = p.n_adapters;
  a.rope = static_cast<const uint8_t*>(rope_table);
  // whole pages of the table only (a page-major table holds positions in blocks of 16)
  a.rope_positions = p.rope_table ? p.rope_table_positions / kPage * kPage : (p.max_seq_len + kPage - 1) / kPage * kPage;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.0f / sqrtf((float)kHeadDim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.kb_map_ok = 0;
  const int64_t kb_pages = (int64_t)p.pools.num_kv_heads * p.pools.num_base_pages;
  PFN_cuTensorMapEncodeTiled_v12000 enc = kb_map_encoder();
  if (enc && kb_pages < (1ll << 31)) {
    const cuuint64_t dims[4] = {128, 16, 2, (cuuint64_t)kb_pages};
    const cuuint64_t strides[3] = {128, 2048, kBaseTile};
    const cuuint32_t box[4] = {128, 16, 1, kBlockPages};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    a.kb_map_ok = enc(&a.kb_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(a.k_base), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const int64_t rows = (int64_t)p.q_len * G;
  dim3 grid((unsigned)((rows + kRows - 1) / kRows), p.n_agents, p.num_kv_heads);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fkv
