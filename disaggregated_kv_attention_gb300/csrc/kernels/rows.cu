// Row scatter into the paged pools and copy-on-write row copies.
//
// forkkv_write_rows: the base activations (xW_k already rotated, xW_v) and the
// residual activations (xA_k, xA_v) of new tokens go to separate pools (ForkKV
// L2 section 7, disaggregation); each 16-byte chunk lands at its swizzled spot.
// forkkv_cow_copy_rows: the pack path of the ForkServe unaligned tail copies
// only the n_valid leading rows of a page (ForkServe README, "Status").
#include "../internal.h"
#include "common.cuh"

namespace fkv {
namespace {

struct WriteArgs {
  uint8_t* k_base;
  uint8_t* v_base;
  uint8_t* k_res;
  uint8_t* v_res;
  int64_t num_base_pages, num_res_pages;
  int32_t hkv, n_rows;
  const int32_t* slot_base;
  const int32_t* slot_res;
  const uint4* kb;
  const uint4* vb;
  const uint4* kr;
  const uint4* vr;
  uint32_t* status;
};

// blockIdx.y == 0: base rows, one thread per 16-byte chunk of (row, head, K|V);
// blockIdx.y == 1: residual rows, one thread per chunk of (row, k|v).
__global__ void __launch_bounds__(256) write_rows_kernel(const WriteArgs a) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.y == 0) {
    if (!a.slot_base) return;
    const int64_t per_row = (int64_t)a.hkv * 32;
    if (idx >= (int64_t)a.n_rows * per_row) return;
    const int32_t row = (int32_t)(idx / per_row);
    const int32_t rem = (int32_t)(idx % per_row);
    const int32_t h = rem >> 5, kv = (rem >> 4) & 1, c = rem & 15;
    const int32_t slot = a.slot_base[row];
    if (slot < 0) return;
    const int64_t page = slot >> 4;
    const int32_t t = slot & 15;
    if (page >= a.num_base_pages) {
      flag_status(a.status, kDevBadPage);
      return;
    }
    const uint4* src = kv ? a.vb : a.kb;
    const uint4 v = src[((int64_t)row * a.hkv + h) * 16 + c];
    uint8_t* dst = (kv ? a.v_base : a.k_base) + ((int64_t)h * a.num_base_pages + page) * kBaseTile + base_off(t, c * 8);
    *reinterpret_cast<uint4*>(dst) = v;
  } else {
    if (!a.slot_res) return;
    if (idx >= (int64_t)a.n_rows * 4) return;
    const int32_t row = (int32_t)(idx >> 2);
    const int32_t kv = (idx >> 1) & 1, c = idx & 1;
    const int32_t slot = a.slot_res[row];
    if (slot < 0) return;
    const int64_t page = slot >> 4;
    const int32_t t = slot & 15;
    if (page >= a.num_res_pages) {
      flag_status(a.status, kDevBadPage);
      return;
    }
    const uint4* src = kv ? a.vr : a.kr;
    const uint4 v = src[(int64_t)row * 2 + c];
    uint8_t* dst = (kv ? a.v_res : a.k_res) + page * kResTile + res_off(t, c * 8);
    *reinterpret_cast<uint4*>(dst) = v;
  }
}

struct CowArgs {
  uint8_t* k_base;
  uint8_t* v_base;
  uint8_t* k_res;
  uint8_t* v_res;
  int64_t base_layer_bytes, res_layer_bytes;
  int64_t num_base_pages;
  int32_t hkv;
};

// blockIdx.x = job, blockIdx.y = layer.  A base row t occupies the two 128-byte
// segments at t*128 and 2048 + t*128 of each (head, page) tile (the swizzle only
// permutes chunks inside a segment), a residual row the 32 bytes at t*32.  Zero
// jobs clear rows n_valid..15 of their page (the unwritten rows of a frozen tail).
__global__ void __launch_bounds__(256) cow_copy_kernel(const CowArgs a, const __grid_constant__ CowJobBatch b) {
  const forkkv_cow_job job = b.jobs[blockIdx.x];
  const int64_t layer = blockIdx.y;
  if (job.kind == FORKKV_JOB_BASE_ZERO || job.kind == FORKKV_JOB_RES_ZERO) {
    const int32_t rows = kPage - job.n_valid;
    if (job.kind == FORKKV_JOB_BASE_ZERO) {
      const int32_t per_tile = rows * 16;  // 16-byte chunks of the cleared rows
      for (int32_t i = threadIdx.x; i < a.hkv * 2 * per_tile; i += blockDim.x) {
        const int32_t tile = i / per_tile, c = i % per_tile;
        const int32_t h = tile >> 1, kv = tile & 1;
        const int32_t t = job.n_valid + (c >> 4), part = (c >> 3) & 1, w = c & 7;
        uint8_t* pool = (kv ? a.v_base : a.k_base) + layer * a.base_layer_bytes;
        *reinterpret_cast<uint4*>(pool + ((int64_t)h * a.num_base_pages + job.dst_page) * kBaseTile + part * 2048 +
                                  t * 128 + w * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      for (int32_t i = threadIdx.x; i < 2 * rows * 2; i += blockDim.x) {
        const int32_t kv = i / (rows * 2), c = i % (rows * 2);
        uint8_t* pool = (kv ? a.v_res : a.k_res) + layer * a.res_layer_bytes;
        *reinterpret_cast<uint4*>(pool + (int64_t)job.dst_page * kResTile + (job.n_valid + (c >> 1)) * 32 +
                                  (c & 1) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }
  if (job.kind == FORKKV_JOB_BASE) {
    const int32_t per_tile = job.n_valid * 16;  // 16-byte chunks of the valid rows
    const int32_t total = a.hkv * 2 * per_tile;
    for (int32_t i = threadIdx.x; i < total; i += blockDim.x) {
      const int32_t tile = i / per_tile, c = i % per_tile;
      const int32_t h = tile >> 1, kv = tile & 1;
      const int32_t t = c >> 4, part = (c >> 3) & 1, w = c & 7;
      const uint32_t off = part * 2048 + t * 128 + w * 16;
      uint8_t* pool = (kv ? a.v_base : a.k_base) + layer * a.base_layer_bytes;
      const int64_t head0 = (int64_t)h * a.num_base_pages;
      const uint4 v = *reinterpret_cast<const uint4*>(pool + (head0 + job.src_page) * kBaseTile + off);
      *reinterpret_cast<uint4*>(pool + (head0 + job.dst_page) * kBaseTile + off) = v;
    }
  } else {
    const int32_t total = 2 * job.n_valid * 2;
    for (int32_t i = threadIdx.x; i < total; i += blockDim.x) {
      const int32_t kv = i / (job.n_valid * 2), c = i % (job.n_valid * 2);
      uint8_t* pool = (kv ? a.v_res : a.k_res) + layer * a.res_layer_bytes;
      const uint32_t off = (c >> 1) * 32 + (c & 1) * 16;
      const uint4 v = *reinterpret_cast<const uint4*>(pool + (int64_t)job.src_page * kResTile + off);
      *reinterpret_cast<uint4*>(pool + (int64_t)job.dst_page * kResTile + off) = v;
    }
  }
}

struct RopeArgs {
  uint32_t turns[128];  // 64 frequencies: 64-bit fixed-point turn fractions, (hi, lo) pairs
  int32_t n_positions;
  uint8_t* table;
};

// One thread per (position, frequency group).  The angle p * f_i is reduced to a
// fraction of a turn exactly in 64-bit integer arithmetic (p * F_i mod 2^64 with
// F_i = f_i / (2 pi) * 2^64), so large positions lose no precision before sin/cos.
__global__ void __launch_bounds__(256) rope_table_kernel(const __grid_constant__ RopeArgs a) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)a.n_positions * 32) return;
  const int32_t p = (int32_t)(idx >> 5), m = (int32_t)(idx & 31);
  float cs[2], sn[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int i = 2 * m + e;
    const uint64_t F = ((uint64_t)a.turns[2 * i] << 32) | a.turns[2 * i + 1];
    const uint64_t frac = (uint64_t)(uint32_t)p * F;          // turns mod 1, in units of 2^-64
    const float y = (float)(int64_t)frac * 0x1p-63f;            // 2 * turns in [-1, 1)
    sincospif(y, &sn[e], &cs[e]);
  }
  uint2 v;
  v.x = pack_bf16(cs[0], cs[1]);
  v.y = pack_bf16(sn[0], sn[1]);
  *reinterpret_cast<uint2*>(a.table + rope_off(p, m)) = v;
}

// Self-test of the bounded waits: one thread waits on a shared-memory mbarrier that nothing
// arrives on, through the same helper every pipeline wait uses, with a poll limit of `polls`.
// The helper gives up, records kDevTimeout and the kernel returns normally.
__global__ void wait_selftest_kernel(uint32_t polls, uint32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
    mbar_wait(&bar, 0, status, polls);
  }
}

}  // namespace

cudaError_t launch_write_rows(const forkkv_pool_desc& pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                              const int32_t* slot_res, const void* kb, const void* vb, const void* kr,
                              const void* vr, uint32_t* status, cudaStream_t stream) {
  if (n_rows == 0) return cudaSuccess;
  WriteArgs a;
  const int64_t base_layer = (int64_t)pools.num_base_pages * pools.num_kv_heads * kBaseTile;
  const int64_t res_layer = (int64_t)pools.num_res_pages * kResTile;
  a.k_base = static_cast<uint8_t*>(pools.k_base) + layer * base_layer;
  a.v_base = static_cast<uint8_t*>(pools.v_base) + layer * base_layer;
  a.k_res = static_cast<uint8_t*>(pools.k_res) + layer * res_layer;
  a.v_res = static_cast<uint8_t*>(pools.v_res) + layer * res_layer;
  a.num_base_pages = pools.num_base_pages;
  a.num_res_pages = pools.num_res_pages;
  a.hkv = pools.num_kv_heads;
  a.n_rows = n_rows;
  a.slot_base = slot_base;
  a.slot_res = slot_res;
  a.kb = static_cast<const uint4*>(kb);
  a.vb = static_cast<const uint4*>(vb);
  a.kr = static_cast<const uint4*>(kr);
  a.vr = static_cast<const uint4*>(vr);
  a.status = status;
  const int64_t work = (int64_t)n_rows * pools.num_kv_heads * 32;
  dim3 grid((unsigned)((work + 255) / 256), 2);
  write_rows_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_cow_copy(const forkkv_pool_desc& pools, const CowJobBatch& batch, cudaStream_t stream) {
  if (batch.n == 0) return cudaSuccess;
  CowArgs a;
  a.k_base = static_cast<uint8_t*>(pools.k_base);
  a.v_base = static_cast<uint8_t*>(pools.v_base);
  a.k_res = static_cast<uint8_t*>(pools.k_res);
  a.v_res = static_cast<uint8_t*>(pools.v_res);
  a.base_layer_bytes = (int64_t)pools.num_base_pages * pools.num_kv_heads * kBaseTile;
  a.res_layer_bytes = (int64_t)pools.num_res_pages * kResTile;
  a.num_base_pages = pools.num_base_pages;
  a.hkv = pools.num_kv_heads;
  cow_copy_kernel<<<dim3(batch.n, pools.n_layers), 256, 0, stream>>>(a, batch);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const uint32_t* turns_hi_lo, int32_t n_positions, void* table, cudaStream_t stream) {
  if (n_positions == 0) return cudaSuccess;
  RopeArgs a;
  for (int i = 0; i < 128; ++i) a.turns[i] = turns_hi_lo[i];
  a.n_positions = n_positions;
  a.table = static_cast<uint8_t*>(table);
  const int64_t work = (int64_t)n_positions * 32;
  rope_table_kernel<<<(unsigned)((work + 255) / 256), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint32_t polls, uint32_t* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(polls, status);
  return cudaGetLastError();
}

}  // namespace fkv
