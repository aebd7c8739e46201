// ResidualAttention decode for sm_103a.
//
// Restates ForkKV L2 sections 4 and 7 (deferred RoPE, associativity of the
// value path, dual-accumulator online softmax) as a split-KV decode:
//
//   split kernel  one CTA per (work item, KV head).  A work item is a run of
//                 logical pages shared by 1, 2, 4 or 8 agents (a trunk of the
//                 fork tree, or one agent's private pages).  A producer warp
//                 streams, per stage, the base K/V tiles of the item's pages
//                 (read ONCE for all agents of the item), every agent's residual
//                 k/v tiles and the rotation-table rows into shared memory with
//                 1-D bulk async copies completing on mbarriers.  Each of the 8
//                 consumer warps owns (agent, page lane) and, per 16-key page:
//                   U      = Kr . B_k[:, hD:(h+1)D]        (mma, 16 keys x 128)
//                   K_lora = RoPE_j(U)                     (fp16x2, registers)
//                   S^T    = Kb . q^T + K_lora . q^T       (mma, keys x heads)
//                   online softmax over keys; acc and acc_r both rescaled
//                   acc^T += Vb^T . P^T ; acc_r^T += Vr^T . P^T   (mma)
//                 Warps of the same agent are merged in shared memory and one
//                 partial (m, l, acc, acc_r) per (item, agent, head) is written.
//   combine       one CTA per (agent, KV head): log-sum-exp merge of the
//                 partials, then out = (acc + acc_r . B_v[:, hD:(h+1)D]) / l,
//                 B_v applied once per query head.
//
// mma.sync m16n8k16 with the keys on M and the (padded) query heads on N keeps
// the padding at 8 columns; movmatrix turns the probability fragment into the
// operand of the value products without a trip through shared memory.
#include <math.h>

#include "../internal.h"
#include "common.cuh"

namespace fkv {
namespace {

constexpr int kWarps = 8;                    // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;  // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kSmemBytes = 227 * 1024;  // the sm_100 family's per-block maximum
constexpr int kHeaderBytes = 4096;           // mbarriers, agent ids, page-id cache
constexpr int kPartCols = kHeadDim + kRank;  // 144 floats per (slot, head, query head)

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
  const int32_t* plan;
  int32_t chunk_pages, chunks;
  int32_t n_agents, max_seq_len, n_slots;
  float* part;
  float* ml;
  uint32_t* status;
};

struct Item {
  int32_t p0, p1, na, wpp, slot_base;
  int32_t agents[8];
};

// Pages per pipeline stage for a group of na agents (8 consumer warps = na x warps-per-agent).
__device__ __forceinline__ int32_t stage_pages(int32_t na) { return na == 8 ? 2 : na == 1 ? 8 : 4; }
// Stage layout: [SP][K tile] [SP][V tile] [SP][16 rotation rows] [na][SP][k_res] [na][SP][v_res]
__device__ __forceinline__ int32_t stage_bytes(int32_t sp, int32_t na) {
  return sp * (2 * kBaseTile + 16 * kRopeRow) + 2 * na * sp * kResTile;
}

__device__ __forceinline__ Item load_item(const DecodeArgs& a) {
  Item it;
  if (a.plan) {
    const int32_t* p = a.plan + (int64_t)blockIdx.x * FORKKV_PLAN_ITEM_INTS;
    it.p0 = p[0];
    it.p1 = p[1];
    it.na = p[2];
    it.wpp = p[3];
#pragma unroll
    for (int i = 0; i < 8; ++i) it.agents[i] = p[4 + i];
    it.slot_base = p[12];
    if (it.na != 1 && it.na != 2 && it.na != 4 && it.na != 8) {
      flag_status(a.status, kDevBadArg);
      it.na = 1;
    }
    it.wpp = 8 / it.na;  // warps per agent
    if (it.slot_base < 0 || it.slot_base + it.na > a.n_slots) {
      flag_status(a.status, kDevBadArg);
      it.p1 = it.p0;  // empty: writes nothing useful, reads nothing
      it.slot_base = -1;
    }
  } else {
    const int32_t agent = blockIdx.x / a.chunks, c = blockIdx.x % a.chunks;
    const int32_t L = min(a.seq_lens[agent], a.max_seq_len);
    const int32_t npg = (L + kPage - 1) / kPage;
    it.p0 = c * a.chunk_pages;
    it.p1 = min(it.p0 + a.chunk_pages, npg);
    it.na = 1;
    it.wpp = 8;
#pragma unroll
    for (int i = 0; i < 8; ++i) it.agents[i] = agent;
    it.slot_base = blockIdx.x;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((uint32_t)it.agents[i] >= (uint32_t)a.n_agents) {
      flag_status(a.status, kDevBadArg);
      it.agents[i] = 0;
      it.p1 = it.p0;
    }
  if (it.p0 < 0 || it.p1 > a.pt_stride) {
    flag_status(a.status, kDevBadArg);
    it.p0 = it.p1 = 0;
  }
  if (it.p1 < it.p0) it.p1 = it.p0;
  return it;
}

__device__ __forceinline__ uint32_t bf2_add(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hadd2(*reinterpret_cast<__nv_bfloat162*>(&a), *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Rotate the pair (lo, hi) = (U_d, U_{d+64}) of two adjacent columns by (cos, sin), bf16x2.
__device__ __forceinline__ void rotate_bf16x2(uint32_t& lo, uint32_t& hi, uint32_t c, uint32_t s) {
  const __nv_bfloat162 L = *reinterpret_cast<__nv_bfloat162*>(&lo), H = *reinterpret_cast<__nv_bfloat162*>(&hi);
  const __nv_bfloat162 C = *reinterpret_cast<__nv_bfloat162*>(&c), S = *reinterpret_cast<__nv_bfloat162*>(&s);
  const __nv_bfloat162 l2 = __hfma2(L, C, __hneg2(__hmul2(H, S)));
  const __nv_bfloat162 h2 = __hfma2(L, S, __hmul2(H, C));
  lo = *reinterpret_cast<const uint32_t*>(&l2);
  hi = *reinterpret_cast<const uint32_t*>(&h2);
}

__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  int32_t* s_agents = reinterpret_cast<int32_t*>(smem + 256);  // [8]
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + 512);     // [16 stages][32] page ids (producer only)
  uint8_t* stages = smem + kHeaderBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const Item it = load_item(a);
  const int na = it.na, wpp = it.wpp;
  const int SP = stage_pages(na);
  const int32_t sbytes = stage_bytes(SP, na);
  const int NS = min(kMaxStages, (kSmemBytes - kHeaderBytes) / sbytes);
  const int n_pages = it.p1 - it.p0;
  const int n_stages = (n_pages + SP - 1) / SP;
  const int32_t v_at = SP * kBaseTile, rope_at = 2 * SP * kBaseTile, kr_at = rope_at + SP * 16 * kRopeRow;
  const int32_t vr_at = kr_at + na * SP * kResTile;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_fence_init();
  }
  if (threadIdx.x < 8) s_agents[threadIdx.x] = it.agents[threadIdx.x];
  __syncthreads();

  const int64_t head_base = (int64_t)h * a.num_base_pages;  // first tile of this head (page-major)
  const int g = lane >> 2, q4 = lane & 3;

  // per-warp partial (consumers): acc^T [d][query head], acc_r^T [k][query head], m, l
  float acc[8][4], accr[4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[mb][e] = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) accr[e] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  if (warp == kWarps) {
    // ------------------------------ producer ------------------------------
    // s_ids[stage % 16][32]: [0, SP) base page ids, [8 + ai*SP + pg] residual page id of agent ai, page pg
    const int32_t lead = s_agents[0];
    int issued = 0;
    bool ok = true;
    for (int s = 0; s < n_stages && ok; ++s) {
      if ((s & 15) == 0) {
        int32_t v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {  // 16 independent loads per lane, all in flight together
          v[i] = -1;
          const int ss = s + i;
          if (ss < n_stages) {
            if (lane < 8) {
              const int pi = it.p0 + ss * SP + lane;
              if (lane < SP && pi < it.p1) v[i] = a.bpt[(int64_t)lead * a.pt_stride + pi];
            } else if (lane < 8 + na * SP) {
              const int ai = (lane - 8) / SP, pg = (lane - 8) % SP;
              const int pi = it.p0 + ss * SP + pg;
              if (pi < it.p1) v[i] = a.rpt[(int64_t)s_agents[ai] * a.pt_stride + pi];
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          int32_t x = v[i];
          const int32_t lim = lane < 8 ? a.num_base_pages : a.num_res_pages;
          if (x != -1 && (uint32_t)x >= (uint32_t)lim) {
            flag_status(a.status, kDevBadPage);
            x = 0;
          }
          s_ids[i * 32 + lane] = x;
        }
        __syncwarp();
      }
      const int slot = s % NS;
      const uint32_t round = s / NS;
      if (s >= NS) ok = mbar_wait(&empty[slot], (round - 1) & 1, a.status);
      if (!ok) break;
      const int pbase = it.p0 + s * SP;
      const int nvp = min(SP, it.p1 - pbase);
      uint8_t* st = stages + (int64_t)slot * sbytes;
      const int32_t* ids = s_ids + (s & 15) * 32;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], nvp * (2 * kBaseTile + 16 * kRopeRow) + na * nvp * 2 * kResTile);
      __syncwarp();
      if (lane < 2) {
        // K (lane 0) or V (lane 1) tiles: one bulk copy per run of consecutive page ids
        const uint8_t* pool = lane == 0 ? a.k_base : a.v_base;
        uint8_t* dst = st + (lane == 0 ? 0 : v_at);
        int r0 = 0;
        for (int pg = 1; pg <= nvp; ++pg) {
          if (pg == nvp || ids[pg] != ids[pg - 1] + 1) {
            bulk_g2s(dst + r0 * kBaseTile, pool + (head_base + ids[r0]) * kBaseTile, (pg - r0) * kBaseTile,
                     &full[slot]);
            r0 = pg;
          }
        }
      } else if (lane == 2) {
        int64_t rrow = (int64_t)pbase * 16;
        if (rrow + 16 * nvp > a.rope_positions) {
          flag_status(a.status, kDevBadArg);
          rrow = 0;
        }
        bulk_g2s(st + rope_at, a.rope + rrow * kRopeRow, nvp * 16 * kRopeRow, &full[slot]);
      } else if (lane >= 8 && lane < 8 + na) {
        // residual k and v tiles of one agent, one copy per run of consecutive page ids
        const int ai = lane - 8;
        const int32_t* rid = ids + 8 + ai * SP;
        int r0 = 0;
        for (int pg = 1; pg <= nvp; ++pg) {
          if (pg == nvp || rid[pg] != rid[pg - 1] + 1) {
            const int64_t src = (int64_t)rid[r0] * kResTile;
            const uint32_t n = (pg - r0) * kResTile;
            bulk_g2s(st + kr_at + (ai * SP + r0) * kResTile, a.k_res + src, n, &full[slot]);
            bulk_g2s(st + vr_at + (ai * SP + r0) * kResTile, a.v_res + src, n, &full[slot]);
            r0 = pg;
          }
        }
      }
      issued = s + 1;
    }
    // Drain: never leave the CTA with bulk copies still in flight.
    for (int s = max(0, issued - NS); s < issued; ++s) mbar_wait(&full[s % NS], (s / NS) & 1, a.status);
  } else {
    // ------------------------------ consumers ------------------------------
    const int ai = warp % na, pl = warp / na;
    const int32_t agent = s_agents[ai];
    const int32_t L = a.seq_lens[agent];
    const int32_t pos = a.positions[agent];
    const int G = a.G;
    if (lane == 0 && pl == 0 && h == 0 && (L < 1 || L > a.max_seq_len || pos < 0 || pos >= L))
      flag_status(a.status, kDevBadArg);
    int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
    if ((uint32_t)adapter >= (uint32_t)a.n_adapters) {
      flag_status(a.status, kDevBadArg);
      adapter = 0;
    }

    // q^T operand fragments (B of m16n8k16: n = query head g, k = d), bf16
    uint32_t qb[8][2];
    {
      const __nv_bfloat16* qrow = a.q + ((int64_t)agent * a.hkv * G + (int64_t)h * G + g) * kHeadDim;
#pragma unroll
      for (int s = 0; s < 8; ++s)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          qb[s][e] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * s + 8 * e + 2 * q4) : 0u;
    }
    // B_k operand fragments (B of m16n8k16: k = rank, n = d within the head)
    uint32_t bk[16][2];
    {
      const __nv_bfloat16* B = a.B_k + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
      const int64_t ld = (int64_t)a.hkv * kHeadDim;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const int n = 8 * t + g;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int k = 8 * e + 2 * q4;
          __nv_bfloat162 v;
          v.x = B[k * ld + n];
          v.y = B[(k + 1) * ld + n];
          bk[t][e] = *reinterpret_cast<uint32_t*>(&v);
        }
      }
    }

    // per-lane shared-memory offsets (loop invariant)
    const int mi = lane >> 3;
    const int lrow = (lane & 7) + (mi & 1) * 8, bsel = mi >> 1;  // A fragments of K (keys x d), Kr
    const int tkey = (lane & 7) + (mi >> 1) * 8, vsel = mi & 1;  // transposed A fragments of V, Vr
    uint32_t kofs[4], vofs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kofs[i] = lrow * 128 + (((2 * i + bsel) ^ (lrow & 7)) << 4);
      vofs[i] = tkey * 128 + (((2 * i + vsel) ^ (tkey & 7)) << 4);
    }
    const uint32_t krofs = res_off(lrow, bsel * 8), vrofs = res_off(tkey, vsel * 8);
    const uint32_t rrow0 = g * kRopeRow + q4 * 8, rrow1 = (g + 8) * kRopeRow + q4 * 8;

    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % NS;
      if (!mbar_wait(&full[slot], (s / NS) & 1, a.status)) break;
      const int pbase = it.p0 + s * SP;
      const int nvp = min(SP, it.p1 - pbase);
      const uint32_t st = smem_u32(stages + (int64_t)slot * sbytes);
      for (int pg = pl; pg < nvp; pg += wpp) {
        const uint32_t sK = st + pg * kBaseTile;
        const uint32_t sV = st + v_at + pg * kBaseTile;
        const uint32_t sR = st + rope_at + pg * 16 * kRopeRow;
        const uint32_t sKr = st + kr_at + (ai * SP + pg) * kResTile;
        const uint32_t sVr = st + vr_at + (ai * SP + pg) * kResTile;
        const int j0 = (pbase + pg) * kPage;

        // full keys K = Kb + RoPE_j(Kr B_k) as A fragments, and S^T = K q^T
        float S0[4] = {0.f, 0.f, 0.f, 0.f}, S1[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t ka0, ka1, ka2, ka3;
        ldsm_x4(sKr + krofs, ka0, ka1, ka2, ka3);
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          float U[4][4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int t = 2 * s4 + (x & 1) + (x >> 1) * 8;  // tiles 2s4, 2s4+1, 2s4+8, 2s4+9
            U[x][0] = U[x][1] = U[x][2] = U[x][3] = 0.f;
            mma_bf16(U[x], ka0, ka1, ka2, ka3, bk[t][0], bk[t][1]);
          }
          uint32_t klo[4], khi[4];  // Kb fragments of k-steps s4 (d < 64) and s4 + 4 (d >= 64)
          ldsm_x4(sK + kofs[s4], klo[0], klo[1], klo[2], klo[3]);
          ldsm_x4(sK + 2048 + kofs[s4], khi[0], khi[1], khi[2], khi[3]);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const uint32_t cofs = ((2 * s4 + x) ^ g) << 5;  // frequency group 4(2s4+x)+q4, swizzled by row
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const uint2 cs = ld_shared_u64(sR + (rr ? rrow1 : rrow0) + cofs);
              uint32_t lo = pack_bf16(U[x][2 * rr], U[x][2 * rr + 1]);
              uint32_t hi = pack_bf16(U[x + 2][2 * rr], U[x + 2][2 * rr + 1]);
              rotate_bf16x2(lo, hi, cs.x, cs.y);
              klo[2 * x + rr] = bf2_add(klo[2 * x + rr], lo);
              khi[2 * x + rr] = bf2_add(khi[2 * x + rr], hi);
            }
          }
          mma_bf16(S0, klo[0], klo[1], klo[2], klo[3], qb[s4][0], qb[s4][1]);
          mma_bf16(S1, khi[0], khi[1], khi[2], khi[3], qb[s4 + 4][0], qb[s4 + 4][1]);
        }
        // mask (only the last pages of an agent need it) + online softmax in base 2
        float sc[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = (S0[e] + S1[e]) * a.scale_log2;
        if (!(j0 + kPage - 1 < L && j0 + kPage - 1 <= pos)) {
          const int ja = j0 + g, jb = j0 + g + 8;
          if (!(ja < L && ja <= pos)) sc[0] = sc[1] = -INFINITY;
          if (!(jb < L && jb <= pos)) sc[2] = sc[3] = -INFINITY;
        }
        float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        // lazy rescale: move the reference maximum only when a score exceeds it by 2^8
        if (__any_sync(0xffffffffu, mx0 > m0 + 8.f || mx1 > m1 + 8.f)) {
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float al0 = mn0 == -INFINITY ? 1.f : exp2f(m0 - mn0);
          const float al1 = mn1 == -INFINITY ? 1.f : exp2f(m1 - mn1);
          l0 *= al0;
          l1 *= al1;
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            acc[mb][0] *= al0;
            acc[mb][1] *= al1;
            acc[mb][2] *= al0;
            acc[mb][3] *= al1;
          }
          accr[0] *= al0;
          accr[1] *= al1;
          accr[2] *= al0;
          accr[3] *= al1;
          m0 = mn0;
          m1 = mn1;
        }
        const float mu0 = m0 == -INFINITY ? 0.f : m0, mu1 = m1 == -INFINITY ? 0.f : m1;
        const float p0 = exp2f(sc[0] - mu0), p2 = exp2f(sc[2] - mu0);
        const float p1 = exp2f(sc[1] - mu1), p3 = exp2f(sc[3] - mu1);
        l0 += p0 + p2;
        l1 += p1 + p3;
        // probabilities as the B operand (k = key, n = query head)
        const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
        const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
        // acc^T += Vb^T . P^T ; acc_r^T += Vr^T . P^T
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(sV + (mb >> 2) * 2048 + vofs[mb & 3], r0, r1, r2, r3);
          mma_bf16(acc[mb], r0, r1, r2, r3, pb0, pb1);
        }
        {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(sVr + vrofs, r0, r1, r2, r3);
          mma_bf16(accr, r0, r1, r2, r3, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
  }
  __syncthreads();  // every warp has left the pipeline: the stage buffers are free

  if (warp < kWarps) {  // park this warp's partial in shared memory
    float* sw = reinterpret_cast<float*>(stages) + warp * 8 * kPartCols;
    float* sml = reinterpret_cast<float*>(stages) + kWarps * 8 * kPartCols + warp * 16;
    const int ga = 2 * q4, gb = 2 * q4 + 1;
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      sw[ga * kPartCols + 16 * mb + g] = acc[mb][0];
      sw[gb * kPartCols + 16 * mb + g] = acc[mb][1];
      sw[ga * kPartCols + 16 * mb + g + 8] = acc[mb][2];
      sw[gb * kPartCols + 16 * mb + g + 8] = acc[mb][3];
    }
    sw[ga * kPartCols + kHeadDim + g] = accr[0];
    sw[gb * kPartCols + kHeadDim + g] = accr[1];
    sw[ga * kPartCols + kHeadDim + g + 8] = accr[2];
    sw[gb * kPartCols + kHeadDim + g + 8] = accr[3];
    if (g == 0) {
      sml[ga * 2] = m0;
      sml[ga * 2 + 1] = l0;
      sml[gb * 2] = m1;
      sml[gb * 2 + 1] = l1;
    }
  }
  __syncthreads();

  // merge the warps of each agent and write one partial per (item, agent, head)
  {
    const int G = a.G;
    const float* sbuf = reinterpret_cast<const float*>(stages);
    const float* smlb = sbuf + kWarps * 8 * kPartCols;
    const int total = it.slot_base < 0 ? 0 : na * G * kPartCols;
    for (int idx = threadIdx.x; idx < total; idx += kThreads) {
      const int ai = idx / (G * kPartCols);
      const int r = idx % (G * kPartCols);
      const int gq = r / kPartCols, col = r % kPartCols;
      float M = -INFINITY;
      for (int p = 0; p < wpp; ++p) M = fmaxf(M, smlb[(p * na + ai) * 16 + gq * 2]);
      float v = 0.f, lsum = 0.f;
      if (M != -INFINITY) {
        for (int p = 0; p < wpp; ++p) {
          const int w = p * na + ai;
          const float wt = exp2f(smlb[w * 16 + gq * 2] - M);
          v += wt * sbuf[w * 8 * kPartCols + gq * kPartCols + col];
          lsum += wt * smlb[w * 16 + gq * 2 + 1];
        }
      }
      const int64_t rec = ((int64_t)(it.slot_base + ai) * a.hkv + h) * G + gq;
      a.part[rec * kPartCols + col] = v;
      if (col == 0) {
        a.ml[rec * 2] = M;
        a.ml[rec * 2 + 1] = lsum;
      }
    }
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
    // Split every agent's pages into `chunks` items of `chunk_pages` pages (a multiple
    // of 8, one page per warp per stage) so that A * chunks * Hkv fills two waves.
    const int32_t max_pages = (p.max_seq_len + kPage - 1) / kPage;
    const int64_t want = 2 * 152;
    int32_t chunks = (int32_t)((want + (int64_t)p.n_agents * p.num_kv_heads - 1) /
                               ((int64_t)p.n_agents * p.num_kv_heads));
    chunks = max(1, min(chunks, (max_pages + 7) / 8));
    int32_t chunk_pages = (max_pages + chunks - 1) / chunks;
    chunk_pages = max(8, (chunk_pages + 7) / 8 * 8);
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
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
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
  a.chunk_pages = g.chunk_pages;
  a.chunks = g.chunks;
  a.n_agents = p.n_agents;
  a.max_seq_len = p.max_seq_len;
  a.n_slots = g.n_slots;
  a.part = reinterpret_cast<float*>(ws);
  a.ml = reinterpret_cast<float*>(ws + g.partial_bytes);
  a.status = status;
  decode_split_kernel<<<dim3(g.n_items, p.num_kv_heads), kThreads, kSmemBytes, stream>>>(a);
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
