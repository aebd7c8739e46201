// Internal launch interface between the C-ABI layer (abi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/forkkv.h"

namespace fkv {

constexpr int kMaxCowJobsPerLaunch = 256;
struct CowJobBatch {
  int32_t n;
  forkkv_cow_job jobs[kMaxCowJobsPerLaunch];
};

uint32_t* device_status_ptr();  // status word of the current device, nullptr on failure

cudaError_t launch_write_rows(const forkkv_pool_desc& pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                              const int32_t* slot_res, const void* kb, const void* vb, const void* kr,
                              const void* vr, uint32_t* status, cudaStream_t stream);
cudaError_t launch_cow_copy(const forkkv_pool_desc& pools, const CowJobBatch& batch, cudaStream_t stream);
cudaError_t launch_rope_table(const uint32_t* turns_hi_lo, int32_t n_positions, void* table, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint32_t polls, uint32_t* status, cudaStream_t stream);
cudaError_t launch_residual_fill(const forkkv_pool_desc& pools, int32_t layer, const void* x, int32_t n_tok,
                                 int32_t hidden, const void* A, int32_t n_ag, const int32_t* slot_res,
                                 uint32_t* status, cudaStream_t stream);
cudaError_t launch_append_rows(const forkkv_pool_desc& pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                               const int32_t* slot_res, const void* kb, const void* vb, const void* x, int32_t hidden,
                               const void* A, int32_t n_adapters, const int32_t* adapter_ids, uint32_t* status,
                               cudaStream_t stream);
int32_t fill_columns_per_cta(int32_t n_tok, int32_t n_ag, int32_t sm_count);

// Decode: partial-result workspace geometry.
struct DecodeGeometry {
  int32_t n_items;        // work items (a unit per item and KV head)
  int32_t n_slots;        // partial slots
  int32_t chunk_pages;    // no-plan mode: pages per item
  int32_t chunks;         // no-plan mode: items per agent
  size_t partial_bytes;   // acc + acc_r floats
  size_t ml_bytes;        // (m, l) floats
  size_t rope_bytes;      // rotation table built in the workspace (0 if the caller gave one)
  size_t total_bytes;
};
DecodeGeometry decode_geometry(const forkkv_attn_params& p);
cudaError_t launch_decode(const forkkv_attn_params& p, const DecodeGeometry& g, const void* rope_table,
                          uint32_t* status, cudaStream_t stream);
cudaError_t launch_prefill(const forkkv_attn_params& p, const void* rope_table, uint32_t* status,
                           cudaStream_t stream);

}  // namespace fkv
