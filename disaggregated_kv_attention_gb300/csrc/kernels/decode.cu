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
constexpr int kHeaderBytes = 1024;           // mbarriers
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

__device__ __forceinline__ int32_t stage_bytes(int32_t wpp) { return wpp * (2 * kBaseTile + 16 * kRopeRow) + 8 * 2 * kResTile; }

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
    it.wpp = 8 / it.na;
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

__global__ void __launch_bounds__(kThreads, 1) decode_split_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint8_t* stages = smem + kHeaderBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const Item it = load_item(a);
  const int na = it.na, wpp = it.wpp;
  const int32_t sbytes = stage_bytes(wpp);
  const int NS = min(kMaxStages, (kSmemBytes - kHeaderBytes) / sbytes);
  const int n_pages = it.p1 - it.p0;
  const int n_stages = (n_pages + wpp - 1) / wpp;
  // stage layout: [wpp][K tile | V tile] [wpp][rotation rows of 16 positions] [8 warps][k_res | v_res]
  const int32_t rope_at = wpp * 2 * kBaseTile;
  const int32_t res_at = rope_at + wpp * 16 * kRopeRow;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int64_t base_tile_stride = (int64_t)a.hkv * kBaseTile;
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
    const int32_t lead = it.agents[0];
    int issued = 0;
    bool ok = true;
    for (int s = 0; s < n_stages && ok; ++s) {
      const int slot = s % NS;
      const uint32_t round = s / NS;
      if (s >= NS) ok = mbar_wait(&empty[slot], (round - 1) & 1, a.status);
      if (!ok) break;
      const int pbase = it.p0 + s * wpp;
      const int nvp = min(wpp, it.p1 - pbase);
      uint8_t* st = stages + (int64_t)slot * sbytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], nvp * (2 * kBaseTile + 16 * kRopeRow) + nvp * na * 2 * kResTile);
      __syncwarp();
      if (lane < nvp) {
        const int pi = pbase + lane;
        int32_t page = a.bpt[(int64_t)lead * a.pt_stride + pi];
        if ((uint32_t)page >= (uint32_t)a.num_base_pages) {
          flag_status(a.status, kDevBadPage);
          page = 0;
        }
        int64_t rrow = (int64_t)pi * 16;
        if (rrow + 16 > a.rope_positions) {
          flag_status(a.status, kDevBadArg);
          rrow = 0;
        }
        const int64_t off = (int64_t)page * base_tile_stride + (int64_t)h * kBaseTile;
        bulk_g2s(st + lane * 2 * kBaseTile, a.k_base + off, kBaseTile, &full[slot]);
        bulk_g2s(st + lane * 2 * kBaseTile + kBaseTile, a.v_base + off, kBaseTile, &full[slot]);
        bulk_g2s(st + rope_at + lane * 16 * kRopeRow, a.rope + rrow * kRopeRow, 16 * kRopeRow, &full[slot]);
      } else if (lane >= 8 && lane < 16) {
        const int w = lane - 8;
        const int ai = w % na, pl = w / na;
        if (pl < nvp) {
          const int pi = pbase + pl;
          int32_t page = a.rpt[(int64_t)it.agents[ai] * a.pt_stride + pi];
          if ((uint32_t)page >= (uint32_t)a.num_res_pages) {
            flag_status(a.status, kDevBadPage);
            page = 0;
          }
          bulk_g2s(st + res_at + w * 2 * kResTile, a.k_res + (int64_t)page * kResTile, kResTile, &full[slot]);
          bulk_g2s(st + res_at + w * 2 * kResTile + kResTile, a.v_res + (int64_t)page * kResTile, kResTile,
                   &full[slot]);
        }
      }
      issued = s + 1;
    }
    // Drain: never leave the CTA with bulk copies still in flight.
    for (int s = max(0, issued - NS); s < issued; ++s) mbar_wait(&full[s % NS], (s / NS) & 1, a.status);
  } else {
    // ------------------------------ consumers ------------------------------
    const int ai = warp % na, pl = warp / na;
    const int32_t agent = it.agents[ai];
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

    // q^T operand fragments (B of m16n8k16: n = query head g, k = d), bf16 and fp16
    uint32_t qb[8][2], qh[8][2];
    {
      const __nv_bfloat16* qrow = a.q + ((int64_t)agent * a.hkv * G + (int64_t)h * G + g) * kHeadDim;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = 16 * s + 8 * e + 2 * q4;
          uint32_t raw = 0;
          if (g < G) raw = *reinterpret_cast<const uint32_t*>(qrow + d);
          qb[s][e] = raw;
          const float2 f = bf2_to_f2(raw);
          qh[s][e] = pack_f16(f.x, f.y);
        }
      }
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

    const int mi = lane >> 3;
    const int lrow = (lane & 7) + (mi & 1) * 8;   // ldmatrix row for the non-transposed A loads
    const int tkey = (lane & 7) + (mi >> 1) * 8;  // ldmatrix row for the transposed loads

    for (int s = 0; s < n_stages; ++s) {
      const int slot = s % NS;
      if (!mbar_wait(&full[slot], (s / NS) & 1, a.status)) break;
      const int pi = it.p0 + s * wpp + pl;
      if (pi < it.p1) {
        const uint8_t* st = stages + (int64_t)slot * sbytes;
        const uint32_t sK = smem_u32(st + pl * 2 * kBaseTile);
        const uint32_t sV = sK + kBaseTile;
        const uint32_t sR = smem_u32(st + rope_at + pl * 16 * kRopeRow);
        const uint32_t sKr = smem_u32(st + res_at + warp * 2 * kResTile);
        const uint32_t sVr = sKr + kResTile;
        const int j0 = pi * kPage;

        float S[4] = {0.f, 0.f, 0.f, 0.f};
        // base scores: S^T += Kb . q^T
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(sK + base_off(lrow, 16 * s8 + (mi >> 1) * 8), r0, r1, r2, r3);
          mma_bf16(S, r0, r1, r2, r3, qb[s8][0], qb[s8][1]);
        }
        // residual keys: up-project, rotate (deferred RoPE), score
        uint32_t ka0, ka1, ka2, ka3;
        ldsm_x4(sKr + res_off(lrow, (mi >> 1) * 8), ka0, ka1, ka2, ka3);
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          float U[4][4];
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const int t = 2 * s4 + (x & 1) + (x >> 1) * 8;  // tiles 2s4, 2s4+1, 2s4+8, 2s4+9
            U[x][0] = U[x][1] = U[x][2] = U[x][3] = 0.f;
            mma_bf16(U[x], ka0, ka1, ka2, ka3, bk[t][0], bk[t][1]);
          }
          uint32_t lo_[2][2], hi_[2][2];  // [tile 2s4 | 2s4+1][row g | g+8]
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            const int m = 4 * (2 * s4 + x) + q4;  // frequency group of d = 8t + 2q4
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int kr = g + 8 * rr;
              const uint2 cs = ld_shared_u64(sR + kr * kRopeRow + rope_off(kr, m));
              const __half2 c = as_h2(cs.x), sn = as_h2(cs.y);
              const __half2 lo = __floats2half2_rn(U[x][2 * rr], U[x][2 * rr + 1]);
              const __half2 hi = __floats2half2_rn(U[x + 2][2 * rr], U[x + 2][2 * rr + 1]);
              lo_[x][rr] = as_u32(__hfma2(lo, c, __hneg2(__hmul2(hi, sn))));
              hi_[x][rr] = as_u32(__hfma2(lo, sn, __hmul2(hi, c)));
            }
          }
          mma_f16(S, lo_[0][0], lo_[0][1], lo_[1][0], lo_[1][1], qh[s4][0], qh[s4][1]);
          mma_f16(S, hi_[0][0], hi_[0][1], hi_[1][0], hi_[1][1], qh[s4 + 4][0], qh[s4 + 4][1]);
        }
        // mask + online softmax (base-2 exponent, scale folded in)
        const int ja = j0 + g, jb = j0 + g + 8;
        const bool va = ja < L && ja <= pos, vb = jb < L && jb <= pos;
        const float s0 = va ? S[0] * a.scale_log2 : -INFINITY;
        const float s1 = va ? S[1] * a.scale_log2 : -INFINITY;
        const float s2 = vb ? S[2] * a.scale_log2 : -INFINITY;
        const float s3 = vb ? S[3] * a.scale_log2 : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
        const float p0 = exp2f(s0 - mu0), p2 = exp2f(s2 - mu0);
        const float p1 = exp2f(s1 - mu1), p3 = exp2f(s3 - mu1);
        l0 = l0 * al0 + p0 + p2;
        l1 = l1 * al1 + p1 + p3;
        m0 = mn0;
        m1 = mn1;
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
        // probabilities as the B operand (k = key, n = query head)
        const uint32_t pb0 = movmatrix_t(pack_bf16(p0, p1));
        const uint32_t pb1 = movmatrix_t(pack_bf16(p2, p3));
        // acc^T += Vb^T . P^T
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(sV + base_off(tkey, 16 * mb + (mi & 1) * 8), r0, r1, r2, r3);
          mma_bf16(acc[mb], r0, r1, r2, r3, pb0, pb1);
        }
        // acc_r^T += Vr^T . P^T
        {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(sVr + res_off(tkey, (mi & 1) * 8), r0, r1, r2, r3);
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

__global__ void __launch_bounds__(128) decode_combine_kernel(const __grid_constant__ CombineArgs a) {
  const int agent = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int G = a.G;
  int32_t s_begin, s_end;
  if (a.csr_off) {
    s_begin = a.csr_off[agent];
    s_end = a.csr_off[agent + 1];
  } else {
    s_begin = agent * a.chunks;
    s_end = s_begin + a.chunks;
  }
  int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
  if ((uint32_t)adapter >= (uint32_t)a.n_adapters) adapter = 0;
  float bv[kRank];
  {
    const __nv_bfloat16* B = a.B_v + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim + d;
#pragma unroll
    for (int k = 0; k < kRank; ++k) bv[k] = __bfloat162float(B[(int64_t)k * a.hkv * kHeadDim]);
  }
  __shared__ float accr_s[kRank];
  if (s_begin < 0 || s_end < s_begin || s_end > a.n_slots) {
    if (d == 0) flag_status(a.status, kDevBadArg);
    s_end = s_begin = 0;
  }
  for (int gq = 0; gq < G; ++gq) {
    float M = -INFINITY;
    for (int i = s_begin; i < s_end; ++i) {
      const int32_t slot = a.csr_off ? a.csr_slots[i] : i;
      if ((uint32_t)slot >= (uint32_t)a.n_slots) continue;
      M = fmaxf(M, a.ml[(((int64_t)slot * a.hkv + h) * G + gq) * 2]);
    }
    float acc = 0.f, accr = 0.f, lsum = 0.f;
    for (int i = s_begin; i < s_end; ++i) {
      const int32_t slot = a.csr_off ? a.csr_slots[i] : i;
      if ((uint32_t)slot >= (uint32_t)a.n_slots) continue;
      const int64_t rec = ((int64_t)slot * a.hkv + h) * G + gq;
      const float m = a.ml[rec * 2];
      if (m == -INFINITY) continue;
      const float wt = exp2f(m - M);
      lsum += wt * a.ml[rec * 2 + 1];
      acc += wt * a.part[rec * kPartCols + d];
      if (d < kRank) accr += wt * a.part[rec * kPartCols + kHeadDim + d];
    }
    __syncthreads();
    if (d < kRank) accr_s[d] = accr;
    __syncthreads();
    float o = acc;
#pragma unroll
    for (int k = 0; k < kRank; ++k) o += accr_s[k] * bv[k];
    o = lsum > 0.f ? o / lsum : 0.f;
    a.out[((int64_t)agent * a.hkv * G + (int64_t)h * G + gq) * kHeadDim + d] = __float2bfloat16_rn(o);
  }
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
  decode_combine_kernel<<<dim3(p.n_agents, p.num_kv_heads), 128, 0, stream>>>(c);
  return cudaGetLastError();
}

}  // namespace fkv
