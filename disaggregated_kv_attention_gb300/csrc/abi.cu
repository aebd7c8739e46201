// C ABI entry points of libforkkv (declared in include/forkkv.h): argument
// validation on the host, then launches of the kernels in kernels/*.cu.
// No C++ exception leaves this file; every entry point returns a status code.
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/forkkv.h"
#include "internal.h"

namespace fkv {

// Device status word: kernels OR FORKKV_DEV_* bits into it; forkkv_get_device_status reads and clears it.
__device__ uint32_t g_device_status;

// Its device address on the current device, looked up once per device ordinal (with that device
// current) and cached.  The address belongs to the device's primary context: it goes stale if the
// process resets the device (cudaDeviceReset), after which the library must not be called again.
uint32_t* device_status_ptr() {
  static std::mutex mu;
  static uint32_t* ptrs[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(p);
  }
  return ptrs[dev];
}

}  // namespace fkv

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int32_t check_pools(const forkkv_pool_desc* p) {
  if (!p) return FORKKV_ERR_INVALID_ARG;
  if (p->num_base_pages < 1 || p->num_res_pages < 1 || p->num_kv_heads < 1 || p->num_kv_heads > 16 ||
      p->n_layers < 1)
    return FORKKV_ERR_INVALID_ARG;
  const void* ptrs[4] = {p->k_base, p->v_base, p->k_res, p->v_res};
  for (const void* q : ptrs)
    if (!q || !aligned(q, 16)) return FORKKV_ERR_INVALID_ARG;
  return FORKKV_OK;
}

int32_t cuda_status(cudaError_t e) { return e == cudaSuccess ? FORKKV_OK : FORKKV_ERR_CUDA; }

int32_t check_attn(const forkkv_attn_params* p, bool decode) {
  if (!p) return FORKKV_ERR_INVALID_ARG;
  if (p->head_dim != FORKKV_HEAD_DIM || p->rank != FORKKV_RANK || p->page_size != FORKKV_PAGE_SIZE)
    return FORKKV_ERR_UNSUPPORTED;
  int32_t rc = check_pools(&p->pools);
  if (rc) return rc;
  if (p->n_agents < 1 || p->num_kv_heads != p->pools.num_kv_heads || p->num_q_heads < 1 ||
      p->num_q_heads % p->num_kv_heads != 0)
    return FORKKV_ERR_INVALID_ARG;
  const int32_t G = p->num_q_heads / p->num_kv_heads;
  if (G > FORKKV_MAX_GROUP) return FORKKV_ERR_UNSUPPORTED;
  if (decode ? p->q_len != 1 : p->q_len < 1) return FORKKV_ERR_INVALID_ARG;
  if (p->layer < 0 || p->layer >= p->pools.n_layers) return FORKKV_ERR_INVALID_ARG;
  if (!p->q || !p->out || !p->bpt || !p->rpt || !p->seq_lens || !p->positions || !p->B_k || !p->B_v)
    return FORKKV_ERR_INVALID_ARG;
  if (!aligned(p->q, 16) || !aligned(p->out, 16) || !aligned(p->B_k, 16) || !aligned(p->B_v, 16))
    return FORKKV_ERR_INVALID_ARG;
  if (p->max_seq_len < 1 || p->pt_stride < 1 ||
      (int64_t)p->pt_stride * FORKKV_PAGE_SIZE < (int64_t)p->max_seq_len)
    return FORKKV_ERR_INVALID_ARG;
  if (p->n_adapters < 1 || !(p->sm_scale >= 0.f)) return FORKKV_ERR_INVALID_ARG;
  const int64_t rope_need = ((int64_t)p->max_seq_len + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE * FORKKV_PAGE_SIZE;
  if (p->rope_table) {
    if (!aligned(p->rope_table, 16) || p->rope_table_positions < rope_need) return FORKKV_ERR_INVALID_ARG;
  } else if (!(p->rope_theta > 0.0) || !std::isfinite(p->rope_theta)) {
    return FORKKV_ERR_INVALID_ARG;
  }
  if (p->plan) {
    if (!decode || p->plan_items < 1 || p->plan_slots < 1 || p->plan_ctas < 1) return FORKKV_ERR_INVALID_ARG;
  }
  return FORKKV_OK;
}

// 64-bit fixed-point turn fractions F_i = f_i / (2 pi) * 2^64 of the 64 rotate-half frequencies.
void rope_turns(double theta, uint32_t out[128]) {
  const long double two_pi = 6.283185307179586476925286766559005768L;
  for (int i = 0; i < 64; ++i) {
    const long double f = powl((long double)theta, -2.0L * i / FORKKV_HEAD_DIM);
    long double turns = f / two_pi;
    turns -= floorl(turns);
    const uint64_t F = (uint64_t)ldexpl(turns, 64);
    out[2 * i] = (uint32_t)(F >> 32);
    out[2 * i + 1] = (uint32_t)(F & 0xffffffffu);
  }
}

}  // namespace

extern "C" {

const char* forkkv_strerror(int32_t code) {
  switch (code) {
    case FORKKV_OK: return "ok";
    case FORKKV_ERR_INVALID_ARG: return "invalid argument";
    case FORKKV_ERR_OUT_OF_PAGES: return "out of pages";
    case FORKKV_ERR_BAD_PAGE: return "page id out of range";
    case FORKKV_ERR_REFCOUNT: return "refcount underflow";
    case FORKKV_ERR_UNSUPPORTED: return "unsupported geometry (needs head_dim 128, rank 16, page 16, group <= 8)";
    case FORKKV_ERR_CUDA: return "CUDA runtime error";
    case FORKKV_ERR_SCRATCH: return "workload needs more scratch than the static decode buffer holds";
    default: return "unknown status";
  }
}

int32_t forkkv_version(void) { return 100; }

int32_t forkkv_write_rows(const forkkv_pool_desc* pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                          const int32_t* slot_res, const void* k_base_rows, const void* v_base_rows,
                          const void* k_res_rows, const void* v_res_rows, void* stream) {
  int32_t rc = check_pools(pools);
  if (rc) return rc;
  if (layer < 0 || layer >= pools->n_layers || n_rows < 0) return FORKKV_ERR_INVALID_ARG;
  if (slot_base && (!k_base_rows || !v_base_rows || !aligned(k_base_rows, 16) || !aligned(v_base_rows, 16)))
    return FORKKV_ERR_INVALID_ARG;
  if (slot_res && (!k_res_rows || !v_res_rows || !aligned(k_res_rows, 16) || !aligned(v_res_rows, 16)))
    return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  return cuda_status(fkv::launch_write_rows(*pools, layer, n_rows, slot_base, slot_res, k_base_rows, v_base_rows,
                                            k_res_rows, v_res_rows, st, as_stream(stream)));
}

int32_t forkkv_residual_fill(const forkkv_pool_desc* pools, int32_t layer, const void* x, int32_t n_tok,
                             int32_t hidden, const void* A, int32_t n_agents, const int32_t* slot_res, void* stream) {
  int32_t rc = check_pools(pools);
  if (rc) return rc;
  if (layer < 0 || layer >= pools->n_layers || n_tok < 0 || n_agents < 0 || n_agents > (1 << 20))
    return FORKKV_ERR_INVALID_ARG;
  if (n_tok == 0 || n_agents == 0) return FORKKV_OK;
  if (!x || !A || !slot_res || !aligned(x, 16) || !aligned(A, 16) || hidden < 8 || hidden % 8 != 0)
    return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  return cuda_status(
      fkv::launch_residual_fill(*pools, layer, x, n_tok, hidden, A, n_agents, slot_res, st, as_stream(stream)));
}

int32_t forkkv_append_rows(const forkkv_pool_desc* pools, int32_t layer, int32_t n_rows, const int32_t* slot_base,
                           const int32_t* slot_res, const void* k_base_rows, const void* v_base_rows, const void* x,
                           int32_t hidden, const void* A, int32_t n_adapters, const int32_t* adapter_ids,
                           void* stream) {
  int32_t rc = check_pools(pools);
  if (rc) return rc;
  if (layer < 0 || layer >= pools->n_layers || n_rows < 0) return FORKKV_ERR_INVALID_ARG;
  if (slot_base && (!k_base_rows || !v_base_rows || !aligned(k_base_rows, 16) || !aligned(v_base_rows, 16)))
    return FORKKV_ERR_INVALID_ARG;
  if (slot_res && (!x || !A || !aligned(x, 16) || !aligned(A, 16) || hidden < 8 || hidden % 8 != 0 ||
                   n_adapters < 1))
    return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  return cuda_status(fkv::launch_append_rows(*pools, layer, n_rows, slot_base, slot_res, k_base_rows, v_base_rows, x,
                                             hidden, A, n_adapters, adapter_ids, st, as_stream(stream)));
}

int32_t forkkv_cow_copy_rows(const forkkv_pool_desc* pools, const forkkv_cow_job* jobs, int32_t n_jobs,
                             void* stream) {
  int32_t rc = check_pools(pools);
  if (rc) return rc;
  if (n_jobs < 0 || (n_jobs > 0 && !jobs)) return FORKKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_jobs; ++i) {
    const forkkv_cow_job& j = jobs[i];
    if (j.kind != FORKKV_JOB_BASE && j.kind != FORKKV_JOB_RES && j.kind != FORKKV_JOB_BASE_ZERO &&
        j.kind != FORKKV_JOB_RES_ZERO)
      return FORKKV_ERR_INVALID_ARG;
    if (j.n_valid < 0 || j.n_valid > FORKKV_PAGE_SIZE) return FORKKV_ERR_INVALID_ARG;
    const bool base = j.kind == FORKKV_JOB_BASE || j.kind == FORKKV_JOB_BASE_ZERO;
    const int32_t lim = base ? pools->num_base_pages : pools->num_res_pages;
    if (j.src_page < 0 || j.src_page >= lim || j.dst_page < 0 || j.dst_page >= lim) return FORKKV_ERR_BAD_PAGE;
  }
  for (int32_t i = 0; i < n_jobs; i += fkv::kMaxCowJobsPerLaunch) {
    static thread_local fkv::CowJobBatch batch;
    batch.n = n_jobs - i < fkv::kMaxCowJobsPerLaunch ? n_jobs - i : fkv::kMaxCowJobsPerLaunch;
    std::memcpy(batch.jobs, jobs + i, sizeof(forkkv_cow_job) * batch.n);
    rc = cuda_status(fkv::launch_cow_copy(*pools, batch, as_stream(stream)));
    if (rc) return rc;
  }
  return FORKKV_OK;
}

int32_t forkkv_rope_table_bytes(int32_t n_positions, size_t* bytes) {
  if (n_positions < 0 || !bytes) return FORKKV_ERR_INVALID_ARG;
  *bytes = (size_t)((n_positions + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE) * FORKKV_PAGE_SIZE * FORKKV_ROPE_ROW_BYTES;
  return FORKKV_OK;
}

int32_t forkkv_rope_table_build(double rope_theta, int32_t n_positions, void* table, void* stream) {
  if (!(rope_theta > 0.0) || !std::isfinite(rope_theta) || n_positions < 0 || (n_positions > 0 && !table) ||
      !aligned(table, 16))
    return FORKKV_ERR_INVALID_ARG;
  uint32_t turns[128];
  rope_turns(rope_theta, turns);
  return cuda_status(fkv::launch_rope_table(turns, n_positions, table, as_stream(stream)));
}

int32_t forkkv_decode_workspace_size(const forkkv_attn_params* p, size_t* bytes) {
  int32_t rc = check_attn(p, true);
  if (rc) return rc;
  if (!bytes) return FORKKV_ERR_INVALID_ARG;
  *bytes = fkv::decode_geometry(*p).total_bytes;
  return FORKKV_OK;
}

int32_t forkkv_residual_attn_decode(const forkkv_attn_params* p, void* stream) {
  int32_t rc = check_attn(p, true);
  if (rc) return rc;
  const fkv::DecodeGeometry g = fkv::decode_geometry(*p);
  if (!p->workspace || !aligned(p->workspace, 256) || p->workspace_bytes < g.total_bytes)
    return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  const void* rope = p->rope_table;
  if (!rope) {
    uint8_t* t = static_cast<uint8_t*>(p->workspace) + g.partial_bytes + g.ml_bytes;
    uint32_t turns[128];
    rope_turns(p->rope_theta, turns);
    const int32_t npos = (p->max_seq_len + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE * FORKKV_PAGE_SIZE;
    rc = cuda_status(fkv::launch_rope_table(turns, npos, t, as_stream(stream)));
    if (rc) return rc;
    rope = t;
  }
  return cuda_status(fkv::launch_decode(*p, g, rope, st, as_stream(stream)));
}

int32_t forkkv_prefill_workspace_size(const forkkv_attn_params* p, size_t* bytes) {
  int32_t rc = check_attn(p, false);
  if (rc) return rc;
  if (!bytes) return FORKKV_ERR_INVALID_ARG;
  *bytes = p->rope_table ? 0
                         : (size_t)((p->max_seq_len + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE * FORKKV_PAGE_SIZE) *
                               FORKKV_ROPE_ROW_BYTES;
  return FORKKV_OK;
}

int32_t forkkv_residual_attn_prefill_chunk(const forkkv_attn_params* p, void* stream) {
  int32_t rc = check_attn(p, false);
  if (rc) return rc;
  size_t need = 0;
  forkkv_prefill_workspace_size(p, &need);
  if (need && (!p->workspace || !aligned(p->workspace, 256) || p->workspace_bytes < need))
    return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  const void* rope = p->rope_table;
  if (!rope) {
    uint32_t turns[128];
    rope_turns(p->rope_theta, turns);
    const int32_t npos = (p->max_seq_len + FORKKV_PAGE_SIZE - 1) / FORKKV_PAGE_SIZE * FORKKV_PAGE_SIZE;
    rc = cuda_status(fkv::launch_rope_table(turns, npos, p->workspace, as_stream(stream)));
    if (rc) return rc;
    rope = p->workspace;
  }
  return cuda_status(fkv::launch_prefill(*p, rope, st, as_stream(stream)));
}

}  // extern "C"

struct forkkv_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" {

int32_t forkkv_step_graph_create(const forkkv_attn_params* params, const forkkv_step_rows* rows, int32_t n_layers,
                                 forkkv_step_graph** out) {
  if (!params || !out || n_layers < 1) return FORKKV_ERR_INVALID_ARG;
  if (!fkv::device_status_ptr()) return FORKKV_ERR_CUDA;  // resolved outside the capture
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return FORKKV_ERR_CUDA;
  int32_t rc = FORKKV_OK;
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(s);
    return FORKKV_ERR_CUDA;
  }
  for (int32_t l = 0; l < n_layers && rc == FORKKV_OK; ++l) {
    const forkkv_attn_params& p = params[l];
    if (rows && rows[l].n_rows > 0) {
      const forkkv_step_rows& r = rows[l];
      rc = forkkv_write_rows(&p.pools, p.layer, r.n_rows, r.slot_base, r.slot_res, r.k_base_rows, r.v_base_rows,
                             r.k_res_rows, r.v_res_rows, s);
    }
    if (rc == FORKKV_OK) rc = forkkv_residual_attn_decode(&p, s);
  }
  const cudaError_t e = cudaStreamEndCapture(s, &graph);  // always: leaves the stream out of capture
  cudaStreamDestroy(s);
  if (rc == FORKKV_OK && e != cudaSuccess) rc = FORKKV_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == FORKKV_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = FORKKV_ERR_CUDA;
  forkkv_step_graph* g = nullptr;
  if (rc == FORKKV_OK) {
    g = new (std::nothrow) forkkv_step_graph();
    if (!g) rc = FORKKV_ERR_INVALID_ARG;
  }
  if (rc != FORKKV_OK) {
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();  // clear a capture error so later calls start clean
    return rc;
  }
  g->graph = graph;
  g->exec = exec;
  *out = g;
  return FORKKV_OK;
}

int32_t forkkv_step_graph_launch(forkkv_step_graph* graph, void* stream) {
  if (!graph || !graph->exec) return FORKKV_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(graph->exec, as_stream(stream)));
}

int32_t forkkv_step_graph_destroy(forkkv_step_graph* graph) {
  if (!graph) return FORKKV_OK;
  cudaError_t e = cudaSuccess;
  if (graph->exec) e = cudaGraphExecDestroy(graph->exec);
  if (graph->graph && e == cudaSuccess) e = cudaGraphDestroy(graph->graph);
  delete graph;
  return cuda_status(e);
}

int32_t forkkv_wait_selftest(uint32_t polls, void* stream) {
  if (polls < 1 || polls > (1u << 20)) return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  return cuda_status(fkv::launch_wait_selftest(polls, st, as_stream(stream)));
}

int32_t forkkv_get_device_status(uint32_t* status, void* stream) {
  if (!status) return FORKKV_ERR_INVALID_ARG;
  uint32_t* st = fkv::device_status_ptr();
  if (!st) return FORKKV_ERR_CUDA;
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, st, sizeof(v), cudaMemcpyDeviceToHost, as_stream(stream));
  if (e == cudaSuccess) e = cudaMemsetAsync(st, 0, sizeof(uint32_t), as_stream(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return FORKKV_ERR_CUDA;
  *status = v;
  return FORKKV_OK;
}

}  // extern "C"
