// Residual rows from hidden states, for sm_103a.
//
// ForkKV L2 section 3 (Figure 6): a child agent forked from a prefix shares the
// prefix's base pages and allocates only residual pages, which hold its own
// rank-16 activations xA_k, xA_v (section 2 Q2: the LoRA projection is
// xW + xA B; the cache keeps xA of each adapter).  Two kernels write them:
//
// residual_fill_kernel: every prefix token for several agents at once.  The
//   agents' down-projections are stacked along N (32 columns per agent: 16 of
//   A_k, then 16 of A_v), so the hidden states x are read once for all of them:
//   R[tok][32 a + c] = x[tok] . W[32 a + c], a dense contraction on the tensor
//   cores (tcgen05, M = 128 tokens, N = 32 g columns, accumulator in tensor
//   memory) fed by 2-D tensor copies (TMA, 128-byte swizzle) through a ring of
//   stages.  The epilogue rounds to bf16 and writes each (agent, token) pair's
//   k and v rows into that agent's residual page.
// append_rows_kernel: one decode token per row, fused with the base-row write:
//   the base rows are scattered as forkkv_write_rows scatters them and the 32
//   residual values x . W[adapter] are computed on the CUDA cores (a matrix-
//   vector product: M = 1 per adapter).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "../internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace fkv {
namespace {

constexpr int kFillM = 128;        // tokens per tile
constexpr int kFillK = 64;         // hidden elements per tensor-copy box (128 bytes of bf16 per row)
constexpr int kFillThreads = 256;  // warp 0 copies, warp 1 issues MMAs, warps 4..7 write rows
constexpr int kFillSmemBudget = 200 * 1024;

struct FillArgs {
  uint8_t* k_res;  // this layer's residual pools
  uint8_t* v_res;
  int64_t num_res_pages;
  const int32_t* slot_res;  // [n_ag][n_tok]
  int32_t n_tok, n_ag, nc, n_kchunks, stages;
  uint32_t tmem_cols;
  uint32_t* status;
};

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// grid (column groups of nc, token tiles): the CTAs that share a token tile are adjacent, so
// the tile's hidden states come from L2 after the first of them has read them.  A stage holds
// kKB boxes of 64 hidden elements of x and of W (kKB * 64 per k-chunk): when the fill is bound by
// HBM, each stage's round trip (copy issue, landing, the MMAs, the release) costs about the same
// whatever its size, so fewer, larger stages move more bytes per round trip.
template <int kKB>
__global__ void __launch_bounds__(kFillThreads, 1)
    residual_fill_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                         const FillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  const uint32_t xbox = kFillM * 128, wbox = (uint32_t)a.nc * 128;
  const uint32_t xbytes = xbox * kKB, wbytes = wbox * kKB, stage_bytes = xbytes + wbytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * stage_bytes);  // full[S], empty[S], done
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * S + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * a.nc, m0 = blockIdx.y * kFillM;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&bars[i], 1);      // the producer's expect_tx arrival
      mbar_init(&bars[S + i], 1);  // the MMA commit that frees the stage
    }
    mbar_init(&bars[2 * S], 1);
    mbar_fence_init();
  }
  if (warp == 1) tc::alloc(s_tmem, a.tmem_cols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tm = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      bool ok = true;
      for (int kc = 0, s = 0, ph = 0; kc < a.n_kchunks && ok; ++kc, ph ^= s + 1 == S, s = s + 1 == S ? 0 : s + 1) {
        if (kc >= S) ok = mbar_wait(&bars[S + s], ph ^ 1, a.status);
        if (!ok) break;
        uint8_t* st = smem + s * stage_bytes;
        mbar_arrive_expect_tx(&bars[s], stage_bytes);
#pragma unroll
        for (int bx = 0; bx < kKB; ++bx) {
          tma_load_2d(st + bx * xbox, &tx, (kc * kKB + bx) * kFillK, m0, &bars[s]);
          tma_load_2d(st + xbytes + bx * wbox, &tw, (kc * kKB + bx) * kFillK, n0, &bars[s]);
        }
      }
      // never leave with copies in flight
      for (int kc = a.n_kchunks - S > 0 ? a.n_kchunks - S : 0; kc < a.n_kchunks && ok; ++kc)
        ok = mbar_wait(&bars[kc % S], (kc / S) & 1, a.status);
    }
    __syncwarp();
  } else if (warp == 1) {
    // the whole warp runs the loop; one elected lane issues the MMAs and commits
    const uint32_t idesc = tc::idesc_bf16(kFillM, a.nc, 0, 0);
    bool ok = true;
    for (int kc = 0, s = 0, ph = 0; kc < a.n_kchunks && ok; ++kc) {
      ok = __all_sync(0xffffffffu, mbar_wait(&bars[s], ph, a.status));
      if (!ok) break;
      tc::fence_after();
      const uint32_t ax = smem_u32(smem + s * stage_bytes), aw = ax + xbytes;
      const uint64_t dx = tc::smem_desc(ax, 16, 1024, tc::kSwizzle128B), dw = tc::smem_desc(aw, 16, 1024, tc::kSwizzle128B);
      if (tc::elect_one()) {
#pragma unroll
        for (int ks = 0; ks < kKB * kFillK / 16; ++ks)  // 16 hidden elements per MMA, 4 per box
          tc::mma_ss(tm, dx + (((ks >> 2) * xbox + 32 * (ks & 3)) >> 4), dw + (((ks >> 2) * wbox + 32 * (ks & 3)) >> 4),
                     idesc, (kc > 0 || ks > 0));
        tc::commit(&bars[S + s]);
      }
      __syncwarp();
      if (++s == S) {
        s = 0;
        ph ^= 1;
      }
    }
    if (tc::elect_one()) tc::commit(&bars[2 * S]);  // the accumulator is final (or the loop gave up: nothing pending)
    __syncwarp();
  } else if (warp >= 4) {
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const int tok = m0 + row;
    const uint32_t tl = tm + ((uint32_t)(32 * q4) << 16);
    const bool ok = mbar_wait(&bars[2 * S], 0, a.status);
    tc::fence_after();
    for (int g = 0; g < a.nc / 32; ++g) {
      uint32_t v[32];
      tc::ld16(tl + 32 * g, v);
      tc::ld16(tl + 32 * g + 16, v + 16);
      tc::wait_ld();
      const int agent = (n0 >> 5) + g;
      if (!ok || tok >= a.n_tok) continue;
      const int32_t slot = a.slot_res[(int64_t)agent * a.n_tok + tok];
      if (slot < 0) continue;
      const int64_t page = slot >> 4;
      const int t = slot & 15;
      if (page >= a.num_res_pages) {
        flag_status(a.status, kDevBadPage);
        continue;
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = pack_bf16(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      uint8_t* kd = a.k_res + page * kResTile;
      uint8_t* vd = a.v_res + page * kResTile;
      *reinterpret_cast<uint4*>(kd + res_off(t, 0)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(kd + res_off(t, 8)) = make_uint4(w[4], w[5], w[6], w[7]);
      *reinterpret_cast<uint4*>(vd + res_off(t, 0)) = make_uint4(w[8], w[9], w[10], w[11]);
      *reinterpret_cast<uint4*>(vd + res_off(t, 8)) = make_uint4(w[12], w[13], w[14], w[15]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tm, a.tmem_cols);
  }
}

struct AppendArgs {
  uint8_t* k_base;
  uint8_t* v_base;
  uint8_t* k_res;
  uint8_t* v_res;
  int64_t num_base_pages, num_res_pages;
  int32_t hkv, hidden, n_adapters;
  const int32_t* slot_base;
  const int32_t* slot_res;
  const uint4* kb;  // [n_rows][hkv][128] bf16
  const uint4* vb;
  const __nv_bfloat16* x;  // [n_rows][hidden]
  const __nv_bfloat16* A;  // [n_adapters][32][hidden]
  const int32_t* adapter_ids;
  uint32_t* status;
};

// One CTA per new token: its base rows (one thread per 16-byte chunk, as forkkv_write_rows) and
// its 32 residual values, warp w computing outputs 4w .. 4w + 3 over the hidden dimension.
__global__ void __launch_bounds__(256) append_rows_kernel(const AppendArgs a) {
  __shared__ uint32_t s_out[16];  // 32 bf16 results: k_res[0..15], v_res[0..15]
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (a.slot_base) {
    const int32_t slot = a.slot_base[row];
    if (slot >= 0) {
      const int64_t page = slot >> 4;
      const int t = slot & 15;
      if (page >= a.num_base_pages) {
        if (threadIdx.x == 0) flag_status(a.status, kDevBadPage);
      } else {
        for (int i = threadIdx.x; i < a.hkv * 32; i += blockDim.x) {
          const int h = i >> 5, kv = (i >> 4) & 1, c = i & 15;
          const uint4 v = (kv ? a.vb : a.kb)[((int64_t)row * a.hkv + h) * 16 + c];
          uint8_t* dst = (kv ? a.v_base : a.k_base) + ((int64_t)h * a.num_base_pages + page) * kBaseTile +
                         base_off(t, c * 8);
          *reinterpret_cast<uint4*>(dst) = v;
        }
      }
    }
  }
  if (!a.slot_res) return;
  int32_t ad = a.adapter_ids ? a.adapter_ids[row] : row;
  if ((uint32_t)ad >= (uint32_t)a.n_adapters) {
    if (threadIdx.x == 0) flag_status(a.status, kDevBadArg);
    ad = 0;
  }
  const __nv_bfloat16* xr = a.x + (int64_t)row * a.hidden;
  const __nv_bfloat16* W = a.A + ((int64_t)ad * 32 + 4 * warp) * a.hidden;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k = 8 * lane; k < a.hidden; k += 8 * 32) {  // hidden is a multiple of 8
    const uint4 xv = *reinterpret_cast<const uint4*>(xr + k);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int o = 0; o < 4; ++o) {
      const uint4 wv = *reinterpret_cast<const uint4*>(W + (int64_t)o * a.hidden + k);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[o] = fmaf(__uint_as_float(xw[i] << 16), __uint_as_float(ww[i] << 16), acc[o]);
        acc[o] = fmaf(__uint_as_float(xw[i] & 0xffff0000u), __uint_as_float(ww[i] & 0xffff0000u), acc[o]);
      }
    }
  }
#pragma unroll
  for (int o = 0; o < 4; ++o)
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) acc[o] += __shfl_xor_sync(0xffffffffu, acc[o], sh);
  if (lane == 0) {
    s_out[2 * warp] = pack_bf16(acc[0], acc[1]);
    s_out[2 * warp + 1] = pack_bf16(acc[2], acc[3]);
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    const int32_t slot = a.slot_res[row];
    if (slot < 0) return;
    const int64_t page = slot >> 4;
    const int t = slot & 15;
    if (page >= a.num_res_pages) {
      if (threadIdx.x == 0) flag_status(a.status, kDevBadPage);
      return;
    }
    const int kv = threadIdx.x >> 1, c = threadIdx.x & 1;
    const uint32_t* src = s_out + 8 * kv + 4 * c;
    *reinterpret_cast<uint4*>((kv ? a.v_res : a.k_res) + page * kResTile + res_off(t, 8 * c)) =
        make_uint4(src[0], src[1], src[2], src[3]);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows][cols] (row stride cols * 2 bytes), tiles of box_rows x 64 columns with
// the 128-byte swizzle; reads past the edges return zeros.
bool encode_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kFillK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int32_t fill_columns_per_cta(int32_t n_tok, int32_t n_ag, int32_t sm_count) {
  // The most agents per CTA (at most 8: N <= 256) whose grid still occupies at least 80 % of
  // the SMs: every column group re-reads the token tile's x (from L2), and a CTA that streams
  // more columns per x tile is the cheaper way to the HBM bound (measured on the 8 x 8192 x
  // 4096 fan-out: 128 columns per CTA in one wave 34 us, 64 columns in 1.7 waves 58 us).
  const int64_t tiles = (n_tok + kFillM - 1) / kFillM;
  int32_t best = 1;
  for (int32_t g = 8; g >= 1; --g)
    if (n_ag % g == 0 && 5 * tiles * (n_ag / g) >= 4 * (int64_t)sm_count) {
      best = g;
      break;
    }
  return 32 * best;
}

cudaError_t launch_residual_fill(const forkkv_pool_desc& pools, int32_t layer, const void* x, int32_t n_tok,
                                 int32_t hidden, const void* A, int32_t n_ag, const int32_t* slot_res,
                                 uint32_t* status, cudaStream_t stream) {
  if (n_tok == 0 || n_ag == 0) return cudaSuccess;
  int dev = 0, sm_count = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int32_t nc = fill_columns_per_cta(n_tok, n_ag, sm_count);
  FillArgs a;
  const int64_t res_layer = (int64_t)pools.num_res_pages * kResTile;
  a.k_res = static_cast<uint8_t*>(pools.k_res) + layer * res_layer;
  a.v_res = static_cast<uint8_t*>(pools.v_res) + layer * res_layer;
  a.num_res_pages = pools.num_res_pages;
  a.slot_res = slot_res;
  a.n_tok = n_tok;
  a.n_ag = n_ag;
  a.nc = nc;
  // two boxes per stage while at least three such stages fit (the HBM-bound shapes: measured
  // 34.2 -> 25.8 us on 8 agents x 8192 tokens x hidden 4096), else one (64 agents x 131072 tokens
  // x hidden 8192, tensor-bound: two stages of two boxes would be slower)
  const int32_t box_pair = kFillM * 128 + nc * 128;
  const int kb = kFillSmemBudget / (2 * box_pair) >= 3 ? 2 : 1;
  a.n_kchunks = (hidden + kFillK * kb - 1) / (kFillK * kb);
  const int32_t stage_bytes = box_pair * kb;
  a.stages = kFillSmemBudget / stage_bytes < 8 ? kFillSmemBudget / stage_bytes : 8;
  a.tmem_cols = nc <= 32 ? 32 : nc <= 64 ? 64 : nc <= 128 ? 128 : 256;
  a.status = status;
  CUtensorMap tx, tw;
  if (!encode_2d(&tx, x, n_tok, hidden, kFillM) || !encode_2d(&tw, A, (int64_t)n_ag * 32, hidden, nc))
    return cudaErrorInvalidValue;
  const int smem = a.stages * stage_bytes + (2 * a.stages + 1) * 8 + 16 + 1024;
  const dim3 grid(n_ag * 32 / nc, (n_tok + kFillM - 1) / kFillM);
  if (kb == 2) {
    e = cudaFuncSetAttribute(residual_fill_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    residual_fill_kernel<2><<<grid, kFillThreads, smem, stream>>>(tx, tw, a);
  } else {
    e = cudaFuncSetAttribute(residual_fill_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    residual_fill_kernel<1><<<grid, kFillThreads, smem, stream>>>(tx, tw, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_append_rows(const forkkv_pool_desc& pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                               const int32_t* slot_res, const void* kb, const void* vb, const void* x, int32_t hidden,
                               const void* A, int32_t n_adapters, const int32_t* adapter_ids, uint32_t* status,
                               cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  AppendArgs a;
  const int64_t base_layer = (int64_t)pools.num_kv_heads * pools.num_base_pages * kBaseTile;
  const int64_t res_layer = (int64_t)pools.num_res_pages * kResTile;
  a.k_base = static_cast<uint8_t*>(pools.k_base) + layer * base_layer;
  a.v_base = static_cast<uint8_t*>(pools.v_base) + layer * base_layer;
  a.k_res = static_cast<uint8_t*>(pools.k_res) + layer * res_layer;
  a.v_res = static_cast<uint8_t*>(pools.v_res) + layer * res_layer;
  a.num_base_pages = pools.num_base_pages;
  a.num_res_pages = pools.num_res_pages;
  a.hkv = pools.num_kv_heads;
  a.hidden = hidden;
  a.n_adapters = n_adapters;
  a.slot_base = slot_base;
  a.slot_res = slot_res;
  a.kb = static_cast<const uint4*>(kb);
  a.vb = static_cast<const uint4*>(vb);
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.A = static_cast<const __nv_bfloat16*>(A);
  a.adapter_ids = adapter_ids;
  a.status = status;
  append_rows_kernel<<<n_rows, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace fkv
