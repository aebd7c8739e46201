// ResidualAttention over a prefill chunk for sm_103a (first version: mma.sync).
//
// Same mathematics as decode (ForkKV L2 sections 4 and 7: deferred RoPE on the
// up-projected residual keys, associativity of the value path, both
// accumulators rescaled together), laid out FlashAttention-style because here
// many query rows share every key tile:
//   grid  (row tile of 128 (token, query-head) rows, agent, KV head)
//   block 8 consumer warps (16 rows each) + 1 producer warp
//   per 64-key stage (4 pages), streamed by bulk async copies:
//     the 8 warps build the stage's full keys once, in shared memory:
//       K = bf16(Kb + RoPE_j(Kr . B_k[:, hD:(h+1)D]))      (up-projection on mma)
//     then each warp:  S = Q K^T, causal mask (key j visible iff j <= position
//     and j < seq_len), online softmax, O += P Vb, O_r += P Vr;
//   epilogue: out = (O + O_r . B_v[:, hD:(h+1)D]) / l, B_v applied once per row.
#include <math.h>

#include "../internal.h"
#include "common.cuh"

namespace fkv {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kRowsPerCta = kWarps * 16;
constexpr int kPagesPerStage = 4;  // 64 keys
constexpr int kStages = 3;
constexpr int kStageBytes = kPagesPerStage * (2 * kBaseTile + 16 * kRopeRow + 2 * kResTile);  // 53248
constexpr int kHeaderBytes = 1024;
constexpr int kKfullBytes = kPagesPerStage * kBaseTile;  // 16 KiB, double buffered
constexpr int kQBytes = kWarps * kBaseTile;               // 128 rows x 128 bf16, 16 rows per warp
constexpr int kSmemBytes = kHeaderBytes + kStages * kStageBytes + 2 * kKfullBytes + kQBytes;

struct PrefillArgs {
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
  const __nv_bfloat16* B_k;
  const __nv_bfloat16* B_v;
  const int32_t* adapter_ids;
  int32_t n_adapters;
  const uint8_t* rope;
  int32_t rope_positions;
  float scale_log2;
  uint32_t* status;
};

// stage layout: [4][K tile | V tile] [4][16 rotation rows] [4][k_res | v_res]
constexpr int kRopeAt = kPagesPerStage * 2 * kBaseTile;
constexpr int kResAt = kRopeAt + kPagesPerStage * 16 * kRopeRow;

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kStages;
  uint64_t* kready = empty + kStages;  // [2]: the 8 warps finished building a full-key buffer
  int32_t* s_meta = reinterpret_cast<int32_t*>(smem + 256);  // [0] = key limit of the CTA
  uint8_t* stages = smem + kHeaderBytes;
  uint8_t* kfull = stages + kStages * kStageBytes;
  uint8_t* qtile = kfull + 2 * kKfullBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q4 = lane & 3;
  const int agent = blockIdx.y, h = blockIdx.z;
  const int G = a.G;
  const int64_t n_rows = (int64_t)a.q_len * G;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
  const int32_t L = min(a.seq_lens[agent], a.max_seq_len);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init(&kready[0], kWarps);
    mbar_init(&kready[1], kWarps);
    mbar_fence_init();
    // keys this CTA may see: up to the largest query position of its rows (and L)
    const int t_first = (int)(row0 / G);
    const int t_last = (int)(min(row0 + kRowsPerCta, n_rows) - 1) / G;
    int32_t pmax = -1;
    for (int t = t_first; t <= t_last; ++t) pmax = max(pmax, a.positions[(int64_t)agent * a.q_len + t]);
    if (a.seq_lens[agent] < 1 || a.seq_lens[agent] > a.max_seq_len) flag_status(a.status, kDevBadArg);
    s_meta[0] = min(pmax + 1, L);
  }
  __syncthreads();
  const int32_t key_limit = s_meta[0];
  const int n_pages = max(0, (key_limit + kPage - 1) / kPage);
  const int n_stages = (n_pages + kPagesPerStage - 1) / kPagesPerStage;
  const int64_t head_base = (int64_t)h * a.num_base_pages * kBaseTile;  // this head's tiles, page-major

  int32_t adapter = a.adapter_ids ? a.adapter_ids[agent] : agent;
  if ((uint32_t)adapter >= (uint32_t)a.n_adapters) {
    if (threadIdx.x == 0) flag_status(a.status, kDevBadArg);
    adapter = 0;
  }

  if (warp == kWarps) {
    // ------------------------------ producer ------------------------------
    int issued = 0;
    bool ok = true;
    for (int s = 0; s < n_stages && ok; ++s) {
      const int slot = s % kStages;
      const uint32_t round = s / kStages;
      if (s >= kStages) ok = mbar_wait(&empty[slot], (round - 1) & 1, a.status);
      if (!ok) break;
      const int pbase = s * kPagesPerStage;
      const int nvp = min(kPagesPerStage, n_pages - pbase);
      uint8_t* st = stages + slot * kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], nvp * (2 * kBaseTile + 16 * kRopeRow + 2 * kResTile));
      __syncwarp();
      if (lane < nvp) {
        const int pi = pbase + lane;
        int32_t bpage = a.bpt[(int64_t)agent * a.pt_stride + pi];
        int32_t rpage = a.rpt[(int64_t)agent * a.pt_stride + pi];
        if ((uint32_t)bpage >= (uint32_t)a.num_base_pages || (uint32_t)rpage >= (uint32_t)a.num_res_pages) {
          flag_status(a.status, kDevBadPage);
          bpage = 0;
          rpage = 0;
        }
        int64_t rrow = (int64_t)pi * 16;
        if (rrow + 16 > a.rope_positions) {
          flag_status(a.status, kDevBadArg);
          rrow = 0;
        }
        const int64_t off = head_base + (int64_t)bpage * kBaseTile;
        bulk_g2s(st + lane * 2 * kBaseTile, a.k_base + off, kBaseTile, &full[slot]);
        bulk_g2s(st + lane * 2 * kBaseTile + kBaseTile, a.v_base + off, kBaseTile, &full[slot]);
        bulk_g2s(st + kRopeAt + lane * 16 * kRopeRow, a.rope + rrow * kRopeRow, 16 * kRopeRow, &full[slot]);
        bulk_g2s(st + kResAt + lane * 2 * kResTile, a.k_res + (int64_t)rpage * kResTile, kResTile, &full[slot]);
        bulk_g2s(st + kResAt + lane * 2 * kResTile + kResTile, a.v_res + (int64_t)rpage * kResTile, kResTile,
                 &full[slot]);
      }
      issued = s + 1;
    }
    for (int s = max(0, issued - kStages); s < issued; ++s) mbar_wait(&full[s % kStages], (s / kStages) & 1, a.status);
    return;  // nothing below involves the producer
  }

  // -------------------------------- consumers --------------------------------
  // rows of this warp: r = row0 + 16*warp + {g, g+8}; row r is (token r / G, query head r % G)
  int32_t rpos[2];
  bool rvalid[2];
  const __nv_bfloat16* qrow[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int64_t r = row0 + 16 * warp + g + 8 * rr;
    rvalid[rr] = r < n_rows;
    const int64_t t = rvalid[rr] ? r / G : 0;
    const int gq = rvalid[rr] ? (int)(r % G) : 0;
    rpos[rr] = rvalid[rr] ? a.positions[(int64_t)agent * a.q_len + t] : -1;
    qrow[rr] = a.q + (((int64_t)agent * a.q_len + t) * a.hkv * G + (int64_t)h * G + gq) * kHeadDim;
  }
  // this warp's 16 query rows, staged once in shared memory (swizzled 16-row tile)
  const uint32_t sQ = smem_u32(qtile + warp * kBaseTile);
  for (int c = lane; c < 16 * 16; c += 32) {
    const int row = c >> 4, ch = c & 15;
    const int64_t r = row0 + 16 * warp + row;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < n_rows) {
      const int64_t t = r / G;
      const int gq = (int)(r % G);
      v = *reinterpret_cast<const uint4*>(a.q + (((int64_t)agent * a.q_len + t) * a.hkv * G + (int64_t)h * G + gq) *
                                                    kHeadDim + ch * 8);
    }
    *reinterpret_cast<uint4*>(qtile + warp * kBaseTile + base_off(row, ch * 8)) = v;
  }
  __syncwarp();
  // B_k fragments for the up-projection tiles this warp builds: tiles 4*hs..4*hs+3 and +8
  const int kp = warp & 3, hs = warp >> 2;
  uint32_t bk[8][2];
  {
    const __nv_bfloat16* B = a.B_k + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
    const int64_t ld = (int64_t)a.hkv * kHeadDim;
#pragma unroll
    for (int x = 0; x < 8; ++x) {
      const int t = 4 * hs + (x & 3) + (x >> 2) * 8;
      const int n = 8 * t + g;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 8 * e + 2 * q4;
        __nv_bfloat162 v;
        v.x = B[k * ld + n];
        v.y = B[(k + 1) * ld + n];
        bk[x][e] = *reinterpret_cast<uint32_t*>(&v);
      }
    }
  }

  float o[16][4], orr[2][4];
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) orr[i][e] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};

  const int mi = lane >> 3;
  const int lrow_a = (lane & 7) + (mi & 1) * 8;  // non-transposed A loads
  const int krow_b = (lane & 7) + (mi >> 1) * 8; // B loads: keys
  const int tkey = (lane & 7) + (mi & 1) * 8;    // transposed B loads: keys

  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % kStages;
    if (!mbar_wait(&full[slot], (s / kStages) & 1, a.status)) break;
    const uint8_t* st = stages + slot * kStageBytes;
    uint8_t* kf = kfull + (s & 1) * kKfullBytes;
    const int pbase = s * kPagesPerStage;
    const int nvp = min(kPagesPerStage, n_pages - pbase);

    // 1. full keys of page kp, column tiles {4hs..4hs+3} and their RoPE partners (+8)
    if (kp < nvp) {
      const uint32_t sKr = smem_u32(st + kResAt + kp * 2 * kResTile);
      const uint32_t sKb = smem_u32(st + kp * 2 * kBaseTile);
      const uint32_t sR = smem_u32(st + kRopeAt + kp * 16 * kRopeRow);
      const uint32_t sKf = smem_u32(kf + kp * kBaseTile);
      uint32_t ka0, ka1, ka2, ka3;
      ldsm_x4(sKr + res_off(lrow_a, (mi >> 1) * 8), ka0, ka1, ka2, ka3);
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        float ulo[4] = {0.f, 0.f, 0.f, 0.f}, uhi[4] = {0.f, 0.f, 0.f, 0.f};
        mma_bf16(ulo, ka0, ka1, ka2, ka3, bk[x][0], bk[x][1]);
        mma_bf16(uhi, ka0, ka1, ka2, ka3, bk[x + 4][0], bk[x + 4][1]);
        const int t = 4 * hs + x;
        const int m = 4 * t + q4;
        const int d = 8 * t + 2 * q4;
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int kr = g + 8 * rr;
          const uint2 cs = ld_shared_u64(sR + kr * kRopeRow + rope_off(kr, m));
          const float2 c = bf2_to_f2(cs.x), sn = bf2_to_f2(cs.y);
          const float l0 = ulo[2 * rr], l1 = ulo[2 * rr + 1], h0 = uhi[2 * rr], h1 = uhi[2 * rr + 1];
          const float2 kbl = bf2_to_f2(ld_shared_u32(sKb + base_off(kr, d)));
          const float2 kbh = bf2_to_f2(ld_shared_u32(sKb + base_off(kr, d + 64)));
          const uint32_t lo = pack_bf16(kbl.x + (l0 * c.x - h0 * sn.x), kbl.y + (l1 * c.y - h1 * sn.y));
          const uint32_t hi = pack_bf16(kbh.x + (h0 * c.x + l0 * sn.x), kbh.y + (h1 * c.y + l1 * sn.y));
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(sKf + base_off(kr, d)), "r"(lo));
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(sKf + base_off(kr, d + 64)), "r"(hi));
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&kready[s & 1]);
    if (!mbar_wait(&kready[s & 1], (s >> 1) & 1, a.status)) break;

    // 2. S = Q K^T over the stage's valid pages
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
    for (int pg = 0; pg < kPagesPerStage; ++pg) {
      if (pg < nvp) {
        const uint32_t sKf = smem_u32(kf + pg * kBaseTile);
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          ldsm_x4(sQ + base_off(lrow_a, 16 * s8 + (mi >> 1) * 8), a0, a1, a2, a3);
          ldsm_x4(sKf + base_off(krow_b, 16 * s8 + (mi & 1) * 8), b0, b1, b2, b3);
          mma_bf16(sc[2 * pg], a0, a1, a2, a3, b0, b1);
          mma_bf16(sc[2 * pg + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    // 3. mask, online softmax (rows g and g+8; four lanes share a row)
    const int kbase = pbase * kPage;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = e >> 1;
        const int j = kbase + 8 * nt + 2 * q4 + (e & 1);
        const bool vis = (nt >> 1) < nvp && j < L && j <= rpos[rr];
        sc[nt][e] = vis ? sc[nt][e] * a.scale_log2 : -INFINITY;
        mx[rr] = fmaxf(mx[rr], sc[nt][e]);
      }
    }
    float alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
      const float mn = fmaxf(mrow[rr], mx[rr]);
      const float mu = mn == -INFINITY ? 0.f : mn;
      alpha[rr] = exp2f(mrow[rr] - mu);
      mrow[rr] = mn;
      mx[rr] = mu;  // reuse as the subtrahend
    }
    float rs[2] = {0.f, 0.f};
    uint32_t pa[4][4];  // P as the A operand, k-step = page
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const float p0 = exp2f(sc[nt][0] - mx[0]), p1 = exp2f(sc[nt][1] - mx[0]);
      const float p2 = exp2f(sc[nt][2] - mx[1]), p3 = exp2f(sc[nt][3] - mx[1]);
      rs[0] += p0 + p1;
      rs[1] += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) lrow[rr] = lrow[rr] * alpha[rr] + rs[rr];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      orr[i][0] *= alpha[0];
      orr[i][1] *= alpha[0];
      orr[i][2] *= alpha[1];
      orr[i][3] *= alpha[1];
    }
    // 4. O += P Vb ; O_r += P Vr
#pragma unroll
    for (int pg = 0; pg < kPagesPerStage; ++pg) {
      if (pg < nvp) {
        const uint32_t sV = smem_u32(st + pg * 2 * kBaseTile + kBaseTile);
        const uint32_t sVr = smem_u32(st + kResAt + pg * 2 * kResTile + kResTile);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + base_off(tkey, 16 * np + (mi >> 1) * 8), b0, b1, b2, b3);
          mma_bf16(o[2 * np], pa[pg][0], pa[pg][1], pa[pg][2], pa[pg][3], b0, b1);
          mma_bf16(o[2 * np + 1], pa[pg][0], pa[pg][1], pa[pg][2], pa[pg][3], b2, b3);
        }
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sVr + res_off(tkey, (mi >> 1) * 8), b0, b1, b2, b3);
        mma_bf16(orr[0], pa[pg][0], pa[pg][1], pa[pg][2], pa[pg][3], b0, b1);
        mma_bf16(orr[1], pa[pg][0], pa[pg][1], pa[pg][2], pa[pg][3], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }

  // epilogue: row sums over the quad, then (O + O_r B_v) / l
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 1);
    lrow[rr] += __shfl_xor_sync(0xffffffffu, lrow[rr], 2);
  }
  // normalise, then add (O_r / l) . B_v[:, hD:(h+1)D] with one fp16 mma per 8 output columns:
  // the O_r fragment (rows x rank) is already the A operand of m16n8k16 (k = rank).
  float inv[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) inv[rr] = lrow[rr] > 0.f ? 1.f / lrow[rr] : 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    o[i][0] *= inv[0];
    o[i][1] *= inv[0];
    o[i][2] *= inv[1];
    o[i][3] *= inv[1];
  }
  const uint32_t ra0 = pack_f16(orr[0][0] * inv[0], orr[0][1] * inv[0]);
  const uint32_t ra1 = pack_f16(orr[0][2] * inv[1], orr[0][3] * inv[1]);
  const uint32_t ra2 = pack_f16(orr[1][0] * inv[0], orr[1][1] * inv[0]);
  const uint32_t ra3 = pack_f16(orr[1][2] * inv[1], orr[1][3] * inv[1]);
  const __nv_bfloat16* Bv = a.B_v + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim;
  const int64_t ld = (int64_t)a.hkv * kHeadDim;
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int n = 8 * nt + g;
    const float b00 = __bfloat162float(Bv[(2 * q4) * ld + n]), b01 = __bfloat162float(Bv[(2 * q4 + 1) * ld + n]);
    const float b10 = __bfloat162float(Bv[(2 * q4 + 8) * ld + n]), b11 = __bfloat162float(Bv[(2 * q4 + 9) * ld + n]);
    mma_f16(o[nt], ra0, ra1, ra2, ra3, pack_f16(b00, b01), pack_f16(b10, b11));
  }
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
    const int d = 8 * nt + 2 * q4;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if (!rvalid[rr]) continue;
      __nv_bfloat16* dst = a.out + (qrow[rr] - a.q) + d;
      *reinterpret_cast<uint32_t*>(dst) = pack_bf16(o[nt][2 * rr], o[nt][2 * rr + 1]);
    }
  }
}

}  // namespace

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
  a.B_k = static_cast<const __nv_bfloat16*>(p.B_k);
  a.B_v = static_cast<const __nv_bfloat16*>(p.B_v);
  a.adapter_ids = p.adapter_ids;
  a.n_adapters = p.n_adapters;
  a.rope = static_cast<const uint8_t*>(rope_table);
  a.rope_positions = p.rope_table ? p.rope_table_positions : (p.max_seq_len + kPage - 1) / kPage * kPage;
  const float scale = p.sm_scale > 0.f ? p.sm_scale : 1.0f / sqrtf((float)kHeadDim);
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  const int64_t rows = (int64_t)p.q_len * G;
  dim3 grid((unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta), p.n_agents, p.num_kv_heads);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fkv
