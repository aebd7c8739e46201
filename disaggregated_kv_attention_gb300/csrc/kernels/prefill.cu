// ResidualAttention over a prefill chunk for sm_103a, on the fifth-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Same mathematics as decode (ForkKV L2 sections 4 and 7: deferred RoPE on the
// up-projected residual keys, associativity of the value path, both
// accumulators rescaled together), laid out for a dense contraction:
//   grid   (tile of 128 (token, query-head) rows, agent, KV head)
//   warps  0      producer: 128-key blocks (8 pages) of K, V, k_res, v_res tiles
//                 into a 2-stage ring with 1-D bulk async copies (one per run of
//                 consecutive page ids)
//          1      allocates 512 TMEM columns; one lane issues every MMA
//          2..5   RoPE group, one key per thread: U = Kr . B_k^T arrives in TMEM;
//                 K = bf16(Kb + RoPE_j(U)) is written to shared memory as the
//                 128-key operand of the next score MMA
//          6..13  softmax group, two warps per query row (half of the keys each):
//                 S from TMEM, causal mask, online softmax; P (bf16) is written
//                 back over S in TMEM
//   MMAs per block:  U[128x128]   = Kr[128x16] . B_k^T           (smem x smem)
//                    S[128x128]   = Q[128x128] . K^T             (smem x smem)
//                    O[128x128]  += P[128x128] . Vb[128x128]      (tmem x smem)
//                    O_r[128x16] += P . Vr[128x16]                (tmem x smem)
//   U, S and P of a block share one of two TMEM buffers (by block parity), so
//   the next block's U, rotation and S run while this block's softmax does;
//   the MMA warp issues, per block, U and S of block b, then P.V of block b - 1.
//   epilogue: out = (O + O_r . B_v[:, hD:(h+1)D]) / l, B_v applied once per row.
// Every wait is on an mbarrier with a bounded spin; a timeout sets the device
// status word instead of hanging.
#include <math.h>

#include "../internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fkv {
namespace {

constexpr int kRows = 128;
constexpr int kBlockPages = 8;
constexpr int kBlockKeys = kBlockPages * kPage;
constexpr int kSoftWarp0 = 6;  // warps 2..5 rotate keys, 6..13 run the softmax
constexpr int kThreads = 14 * 32;

// shared memory (offsets from a 1024-byte aligned base)
constexpr int kOffPmax = 1024;                  // [2 parities][2 halves][128 rows] partial row maxima
constexpr int kOffQ = 3072;                     // Q, K-major 128B-swizzled [2][128 rows][128 B]
constexpr int kOffKF = kOffQ + 32768;           // full keys of one block, same layout
constexpr int kOffStage = kOffKF + 32768;       // 2 stages
constexpr int kStageBytes = 73728;
constexpr int kStK = 0, kStV = 32768, kStKR = 65536, kStVR = 69632;  // 8 K tiles, 8 V tiles, 8 k_res, 8 v_res
constexpr int kOffBk = kOffStage + 2 * kStageBytes;  // B_k^T, K-major 32B-swizzled [128 d][16 r]
constexpr int kOffBv = kOffBk + 4096;                // B_v slice [16][128] bf16
constexpr int kSmemBytes = kOffBv + 4096 + 1024;     // + slack for aligning the base
static_assert(kSmemBytes <= 227 * 1024, "more shared memory than a CTA may have");

// tensor memory columns: two buffers (U, then S, then P over S) by block parity, O, O_r
constexpr uint32_t kTmBuf = 0, kTmO = 256, kTmOr = 384, kTmCols = 512;

// mbarrier indices
enum { kFull0, kFull1, kEmpty0, kEmpty1, kUFull0, kUFull1, kKFReady, kKFFree, kSFull0, kSFull1, kPFull0, kPFull1,
       kPVDone0, kPVDone1, kQReady, kBkReady, kMmaDone, kNumBars };
static_assert(kNumBars * 8 <= 256, "barriers overlap the state that follows them");

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


__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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

  if (threadIdx.x == 0) {
    mbar_init(&bars[kFull0], 1);
    mbar_init(&bars[kFull1], 1);
    mbar_init(&bars[kEmpty0], 5);  // 4 RoPE warps + the MMA commit after the value products
    mbar_init(&bars[kEmpty1], 5);
    mbar_init(&bars[kUFull0], 1);
    mbar_init(&bars[kUFull1], 1);
    mbar_init(&bars[kKFReady], 4);
    mbar_init(&bars[kKFFree], 1);
    mbar_init(&bars[kSFull0], 1);
    mbar_init(&bars[kSFull1], 1);
    mbar_init(&bars[kPFull0], 8);  // every softmax warp
    mbar_init(&bars[kPFull1], 8);
    mbar_init(&bars[kPVDone0], 1);
    mbar_init(&bars[kPVDone1], 1);
    mbar_init(&bars[kQReady], 8);
    mbar_init(&bars[kBkReady], 4);
    mbar_init(&bars[kMmaDone], 1);
    mbar_fence_init();
    // keys this CTA may see: up to the largest query position of its rows (and L)
    const int t_first = (int)(row0 / G);
    const int t_last = (int)((min(row0 + kRows, n_rows) - 1) / G);
    int32_t pmax = -1;
    for (int t = t_first; t <= t_last; ++t) pmax = max(pmax, a.positions[(int64_t)agent * a.q_len + t]);
    if (a.seq_lens[agent] < 1 || a.seq_lens[agent] > a.max_seq_len) flag_status(a.status, kDevBadArg);
    if ((uint32_t)(a.adapter_ids ? a.adapter_ids[agent] : agent) >= (uint32_t)a.n_adapters)
      flag_status(a.status, kDevBadArg);
    s_meta[0] = max(0, min(pmax + 1, L));
  }
  if (warp == 1) tc::alloc(s_tmem, kTmCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = *s_tmem;
  const int32_t key_limit = s_meta[0];
  const int n_pages = (key_limit + kPage - 1) / kPage;
  const int n_blocks = (n_pages + kBlockPages - 1) / kBlockPages;
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sKF = smem + kOffKF;
  uint8_t* sBk = smem + kOffBk;
  uint8_t* sBv = smem + kOffBv;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    const int64_t head_base = (int64_t)h * a.num_base_pages;
    for (int b = 0; b < n_blocks; ++b) {
      const int stage = b & 1;
      if (b >= 2 && !mbar_wait(&bars[kEmpty0 + stage], ((b >> 1) - 1) & 1, a.status)) break;
      const int pbase = b * kBlockPages;
      const int nvp = min(kBlockPages, n_pages - pbase);
      int32_t id = 0;
      if (lane < nvp) {
        id = a.bpt[(int64_t)agent * a.pt_stride + pbase + lane];
        if ((uint32_t)id >= (uint32_t)a.num_base_pages) {
          flag_status(a.status, kDevBadPage);
          id = 0;
        }
      } else if (lane >= 8 && lane - 8 < nvp) {
        id = a.rpt[(int64_t)agent * a.pt_stride + pbase + lane - 8];
        if ((uint32_t)id >= (uint32_t)a.num_res_pages) {
          flag_status(a.status, kDevBadPage);
          id = 0;
        }
      }
      int32_t ids[8];
      const int src0 = lane < 2 ? 0 : 8;  // lanes 0, 1: base page ids; lanes 2, 3: residual page ids
#pragma unroll
      for (int pg = 0; pg < 8; ++pg) ids[pg] = __shfl_sync(0xffffffffu, id, src0 + pg);
      uint8_t* st = smem + kOffStage + stage * kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(&bars[kFull0 + stage], nvp * (2 * kBaseTile + 2 * kResTile));
      __syncwarp();
      if (lane < 4) {
        const uint8_t* pool = lane == 0 ? a.k_base + head_base * kBaseTile
                              : lane == 1 ? a.v_base + head_base * kBaseTile
                              : lane == 2 ? a.k_res : a.v_res;
        uint8_t* dst = st + (lane == 0 ? kStK : lane == 1 ? kStV : lane == 2 ? kStKR : kStVR);
        const uint32_t tile = lane < 2 ? kBaseTile : kResTile;
        int r0 = 0;
        int32_t start = ids[0];
#pragma unroll
        for (int pg = 1; pg <= 8; ++pg) {
          if (pg <= nvp) {
            const bool end = pg == nvp || ids[pg < 8 ? pg : 7] != ids[pg - 1] + 1;
            if (end) {
              bulk_g2s(dst + r0 * tile, pool + (int64_t)start * tile, (pg - r0) * tile, &bars[kFull0 + stage]);
              r0 = pg;
              start = ids[pg < 8 ? pg : 7];
            }
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // Per block b: U(b) into buffer b % 2 (once P.V of block b - 2 is done with it), S(b)
    // over U(b) once the rotation group has built K(b), then P.V of block b - 1.
    if (lane == 0) {
      const uint32_t idU = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idS = tc::idesc_bf16(128, 128, 0, 0);
      const uint32_t idPV = tc::idesc_bf16(128, 128, 0, 1);
      const uint32_t idPVr = tc::idesc_bf16(128, 16, 0, 1);
      const uint32_t aQ = smem_u32(sQ), aKF = smem_u32(sKF), aBk = smem_u32(sBk);
      bool ok = mbar_wait(&bars[kQReady], 0, a.status) && mbar_wait(&bars[kBkReady], 0, a.status);
      // P.V of block c: A = P from its buffer (keys 0..63 at columns 0..31, keys 64..127 at 64..95)
      auto issue_pv = [&](int c) {
        const uint32_t buf = tm + kTmBuf + 128 * (c & 1);
        const uint32_t st = smem_u32(smem + kOffStage + (c & 1) * kStageBytes);
        const int nvp = min(kBlockPages, n_pages - c * kBlockPages);
        for (int ks = 0; ks < nvp; ++ks)
          tc::mma_ts(tm + kTmO, buf + (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4)),
                     tc::smem_desc(st + kStV + ks * kBaseTile, 2048, 1024, tc::kSwizzle128B), idPV, (c > 0 || ks > 0));
        for (int ks = 0; ks < nvp; ++ks)
          tc::mma_ts(tm + kTmOr, buf + (ks < 4 ? 8 * ks : 64 + 8 * (ks - 4)),
                     tc::smem_desc(st + kStVR + ks * kResTile, 4096, 256, tc::kSwizzle32B), idPVr, (c > 0 || ks > 0));
        tc::commit(&bars[kPVDone0 + (c & 1)]);
        tc::commit(&bars[kEmpty0 + (c & 1)]);
      };
      for (int b = 0; b < n_blocks && ok; ++b) {
        const int stage = b & 1;
        const uint32_t st = smem_u32(smem + kOffStage + stage * kStageBytes);
        const uint32_t buf = tm + kTmBuf + 128 * stage;
        ok = mbar_wait(&bars[kFull0 + stage], (b >> 1) & 1, a.status) &&
             (b < 2 || mbar_wait(&bars[kPVDone0 + stage], ((b >> 1) - 1) & 1, a.status));
        if (!ok) break;
        tc::fence_after();
        tc::mma_ss(buf, tc::smem_desc(st + kStKR, 16, 256, tc::kSwizzle32B), tc::smem_desc(aBk, 16, 256, tc::kSwizzle32B),
                   idU, 0);
        tc::commit(&bars[kUFull0 + stage]);
        ok = mbar_wait(&bars[kKFReady], b & 1, a.status);
        if (!ok) break;
        tc::fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          tc::mma_ss(buf, tc::smem_desc(aQ + off, 16, 1024, tc::kSwizzle128B),
                     tc::smem_desc(aKF + off, 16, 1024, tc::kSwizzle128B), idS, ks > 0);
        }
        tc::commit(&bars[kSFull0 + stage]);
        tc::commit(&bars[kKFFree]);
        if (b > 0) {
          ok = mbar_wait(&bars[kPFull0 + ((b - 1) & 1)], ((b - 1) >> 1) & 1, a.status);
          if (!ok) break;
          tc::fence_after();
          issue_pv(b - 1);
        }
      }
      if (ok && n_blocks > 0) {
        ok = mbar_wait(&bars[kPFull0 + ((n_blocks - 1) & 1)], ((n_blocks - 1) >> 1) & 1, a.status);
        if (ok) {
          tc::fence_after();
          issue_pv(n_blocks - 1);
        }
      }
      // never leave with MMAs in flight
      tc::commit(&bars[kMmaDone]);
      mbar_wait(&bars[kMmaDone], 0, a.status);
    }
    __syncwarp();
  } else if (warp < kSoftWarp0) {
    // ------------------------------ RoPE group ------------------------------
    const int row = 32 * (warp & 3) + lane;  // key row of the block == TMEM lane
    const uint32_t tl = tm + ((uint32_t)(32 * (warp & 3)) << 16);
    {  // B_k^T: row d, 16 ranks
      const __nv_bfloat16* B = a.B_k + (int64_t)adapter * kRank * a.hkv * kHeadDim + (int64_t)h * kHeadDim + row;
#pragma unroll
      for (int k = 0; k < kRank; ++k)
        *reinterpret_cast<__nv_bfloat16*>(sBk + tc::sw32_off(row, k)) = B[(int64_t)k * a.hkv * kHeadDim];
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBkReady]);
    }
    const int p = row >> 4, t = row & 15;
    bool ok = true;
    for (int b = 0; b < n_blocks && ok; ++b) {
      const int stage = b & 1;
      uint8_t* st = smem + kOffStage + stage * kStageBytes;
      const uint32_t ub = tl + kTmBuf + 128 * stage;
      const int j = b * kBlockKeys + row;
      // this key's rotation row: logical 32-byte unit u sits at unit u ^ (j % 8)
      uint4 rp[8][2];
      {
        const int jr = j < a.rope_positions ? j : 0;
        const uint4* rrow = reinterpret_cast<const uint4*>(a.rope + (int64_t)jr * kRopeRow);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          rp[u][0] = rrow[(u ^ (j & 7)) * 2];
          rp[u][1] = rrow[(u ^ (j & 7)) * 2 + 1];
        }
      }
      ok = mbar_wait(&bars[kFull0 + stage], (b >> 1) & 1, a.status) &&
           mbar_wait(&bars[kUFull0 + stage], (b >> 1) & 1, a.status);
      if (ok && b > 0) ok = mbar_wait(&bars[kKFFree], (b - 1) & 1, a.status);  // S(b - 1) is done with sKF
      if (!ok) break;
      tc::fence_after();
      const uint8_t* kt = st + kStK + p * kBaseTile;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        uint32_t ulo[16], uhi[16];
        tc::ld16(ub + c, ulo);
        tc::ld16(ub + 64 + c, uhi);
        uint4 kl[2], kh[2];
        kl[0] = *reinterpret_cast<const uint4*>(kt + base_off(t, c));
        kl[1] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 8));
        kh[0] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 64));
        kh[1] = *reinterpret_cast<const uint4*>(kt + base_off(t, c + 72));
        tc::wait_ld();
        const uint32_t* klw = reinterpret_cast<const uint32_t*>(kl);
        const uint32_t* khw = reinterpret_cast<const uint32_t*>(kh);
        uint32_t olo[8], ohi[8];
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {  // elements d = c + 2*i2, c + 2*i2 + 1 (and + 64)
          const int m = (c >> 1) + i2;     // frequency group
          const uint4 w = rp[m >> 2][(m & 3) >> 1];
          const uint32_t cw = (m & 1) ? w.z : w.x, sw = (m & 1) ? w.w : w.y;
          const float lo0 = __uint_as_float(ulo[2 * i2]), lo1 = __uint_as_float(ulo[2 * i2 + 1]);
          const float hi0 = __uint_as_float(uhi[2 * i2]), hi1 = __uint_as_float(uhi[2 * i2 + 1]);
          const float c0 = bf_lo(cw), c1 = bf_hi(cw), s0 = bf_lo(sw), s1 = bf_hi(sw);
          const float kl0 = bf_lo(klw[i2]) + (lo0 * c0 - hi0 * s0);
          const float kl1 = bf_hi(klw[i2]) + (lo1 * c1 - hi1 * s1);
          const float kh0 = bf_lo(khw[i2]) + (hi0 * c0 + lo0 * s0);
          const float kh1 = bf_hi(khw[i2]) + (hi1 * c1 + lo1 * s1);
          olo[i2] = pack_bf16(kl0, kl1);
          ohi[i2] = pack_bf16(kh0, kh1);
        }
        *reinterpret_cast<uint4*>(sKF + tc::sw128_off(128, row, c)) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
        *reinterpret_cast<uint4*>(sKF + tc::sw128_off(128, row, c + 8)) = make_uint4(olo[4], olo[5], olo[6], olo[7]);
        *reinterpret_cast<uint4*>(sKF + tc::sw128_off(128, row, c + 64)) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
        *reinterpret_cast<uint4*>(sKF + tc::sw128_off(128, row, c + 72)) = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      }
      tc::fence_before();
      // keys past the sequence: zero their value rows so that 0 * (never-written data) stays 0
      const int nvp = min(kBlockPages, n_pages - b * kBlockPages);
      if (j >= L && p < nvp) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int ch = 0; ch < 16; ++ch)
          *reinterpret_cast<uint4*>(st + kStV + p * kBaseTile + base_off(t, ch * 8)) = z;
        *reinterpret_cast<uint4*>(st + kStVR + p * kResTile + res_off(t, 0)) = z;
        *reinterpret_cast<uint4*>(st + kStVR + p * kResTile + res_off(t, 8)) = z;
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kKFReady]);
        mbar_arrive(&bars[kEmpty0 + stage]);
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
    const int64_t orow = (((int64_t)agent * a.q_len + tq) * a.hkv * G + (int64_t)h * G + gq) * kHeadDim;
    {  // this half of the Q row into the K-major swizzled tile; this half of the B_v slice
      const uint4* src = reinterpret_cast<const uint4*>(a.q + orow);
#pragma unroll
      for (int ch = 8 * sh; ch < 8 * sh + 8; ++ch) {
        const uint4 v = valid ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sQ + tc::sw128_off(128, qr, ch * 8)) = v;
      }
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
      float bm = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t v0[16], v1[16];
        tc::ld16(tl + buf + 64 * sh + c, v0);
        tc::ld16(tl + buf + 64 * sh + c + 16, v1);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int j = kbase + c + i;
          const float s = __uint_as_float(i < 16 ? v0[i] : v1[i - 16]) * a.scale_log2;
          if (j < L && j <= pos) bm = fmaxf(bm, s);
        }
      }
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
      // P over this half's S columns: keys 64 sh + 2 i, 2 i + 1 at column 64 sh + i
#pragma unroll
      for (int c = 0; c < 64; c += 32) {
        uint32_t v0[16], v1[16], pw[16];
        tc::ld16(tl + buf + 64 * sh + c, v0);
        tc::ld16(tl + buf + 64 * sh + c + 16, v1);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float pr[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int ii = 2 * i + e;
            const int j = kbase + c + ii;
            const float s = __uint_as_float(ii < 16 ? v0[ii] : v1[ii - 16]) * a.scale_log2;
            pr[e] = (j < L && j <= pos) ? exp2f(s - mu) : 0.f;
            l += pr[e];
          }
          pw[i] = pack_bf16(pr[0], pr[1]);
        }
        tc::st16(tl + buf + 64 * sh + (c >> 1), pw);  // over columns of S this thread already read
      }
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
  dim3 grid((unsigned)((rows + kRows - 1) / kRows), p.n_agents, p.num_kv_heads);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fkv
