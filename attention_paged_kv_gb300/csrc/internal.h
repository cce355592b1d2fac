// Host-side internals shared by the planner, the C ABI and the launchers.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"

namespace pa {

// Planner result: the metadata blob (int32 words, the exact bytes copied to
// the start of the workspace) plus the sizes the launchers need.
struct HostPlan {
  std::vector<int32_t> blob;
  int32_t B = 0, Hq = 0, Hkv = 0, D = 0, ps = 0, num_pages = 0, dtype = 0, causal = 1, T = 0, nnz = 0;
  int32_t n_dec = 0, n_pre = 0, n_merge = 0, n_part = 0, G = 1, num_sms = 0;
  int32_t dec_cores = 0;                  // 1: decode items run on the CUDA-core kernel
  int32_t pre_tiles = 2;                  // 128-row Q tiles per prefill item (1 or 2)
  int32_t hnd = 0;                        // cache layout: 0 NHD, 1 HND
  int32_t wait_limit_cycles = 0;          // > 0: bound of each pipeline wait (test hook)
  int32_t n_dec_class[4] = {0, 0, 0, 0};  // decode items per row class, consecutive in item order
  size_t blob_bytes = 0, off_part_o = 0, off_part_lse = 0, total_bytes = 0;
  size_t off_pages = 0, off_req = 0, off_dec = 0, off_pre = 0, off_merge = 0;
  std::vector<int64_t> kv_len;  // per request (debug gather sizes)
};

struct PlanInputs {
  const int32_t* qo_indptr;
  const int32_t* kv_page_indptr;
  const int32_t* kv_page_indices;
  const int32_t* kv_last_page_len;
  int32_t B, Hq, Hkv, D, ps, num_pages, dtype, causal;
  int32_t num_sms, force_prefill, decode_chunk_pages, prefill_chunk_tiles, decode_cuda_cores, kv_layout;
  int32_t prefill_q_tiles;  // 0: the planner's choice, else 1 or 2 Q tiles per prefill item
  int32_t wait_limit_cycles;  // > 0: bound of each pipeline wait in clock cycles (test hook)
  // shared-prefix cascade (n_groups == 0: a plain plan)
  const int32_t* group_indptr;
  const int32_t* prefix_page_indptr;
  const int32_t* prefix_page_indices;
  int32_t n_groups;
};

// Validate and partition; on failure returns the status and fills `err`.
pagedattn_status build_plan(const PlanInputs& in, HostPlan* out, std::string* err);

// Launchers (one per kernel family).  All are asynchronous on `stream`.
struct RunArgs {
  const HostPlan* hp;
  void* workspace;  // device base of the metadata
  const void* q;
  const void* kv;
  void* out;
  float* lse;
  cudaStream_t stream;
  int force_cp_async;
};

cudaError_t launch_prefill(const RunArgs& a, const CUtensorMap* map_sw128, const CUtensorMap* map_q,
                           const CUtensorMap* map_o);  // map_o: [2], 128-row and 32-row boxes over out
cudaError_t launch_decode(const RunArgs& a, const CUtensorMap* map_rows);
cudaError_t launch_merge(const RunArgs& a);
cudaError_t launch_debug_gather(const RunArgs& a, int32_t* page_out, int32_t* slot_out);

// Raise `func`'s dynamic shared memory limit to `bytes` on the current
// device, once per device: the attribute is per device, so `done` keeps one
// bit per device ordinal.  Concurrent first calls may both set it (harmless).
inline cudaError_t set_smem_once(std::atomic<uint64_t>& done, const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch `kernel` on `stream` with programmatic stream serialization: it may
// begin (and run its prologue) while the previous kernel on the stream
// finishes; the kernel itself waits (pdl_wait) before touching data that
// kernel may produce or read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  std::memset(attr, 0, sizeof(attr));
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
#ifndef PA_NO_PDL
  attr[0].val.programmaticStreamSerializationAllowed = 1;
#endif
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Error reporting into the thread-local last-error text (api.cu).
pagedattn_status set_err(pagedattn_status s, const std::string& msg);
pagedattn_status cuda_err(cudaError_t e, const char* what);

// Tensor map over the cache viewed as (D, Hkv, page_size, 2 * num_pages),
// box {box0, 1, box2, 1} (api.cu).
pagedattn_status encode_kv_map(CUtensorMap* m, const HostPlan& hp, const void* kv, uint32_t box0, uint32_t box2,
                               CUtensorMapSwizzle sw);
// Tensor map over q, or over out (same shape), viewed as (D, Hq, T), box
// {64, G, 128 / G}: one 128-row query tile of 64 columns (api.cu).
pagedattn_status encode_q_map(CUtensorMap* m, const HostPlan& hp, const void* q, uint32_t box_rows = 128);

}  // namespace pa

// The plan handle behind pagedattn_plan_t.
struct pagedattn_plan_s {
  pa::HostPlan hp;
  void* workspace = nullptr;
  size_t workspace_bytes = 0;
  int device = -1;
  int force_cp_async = 0;
  // guards the tensor-map cache below: a plan may be run from several host threads
  std::mutex maps_mu;
  // tensor maps over the last kv_cache pointer seen by run()
  const void* map_kv = nullptr;
  CUtensorMap map_rows;   // decode: box {64, 1, min(ps, 64), 1}, 128-byte swizzle (page_size >= 8)
  CUtensorMap map_sw128;  // prefill: box {64, 1, ps, 1}, 128-byte swizzle
  // tensor map over the last q pointer seen by run() (prefill Q tiles)
  const void* map_q_ptr = nullptr;
  CUtensorMap map_q;
  const void* map_o_ptr = nullptr;  // the out array of map_o: 128-row boxes (as map_q), then 32-row boxes
  CUtensorMap map_o[2];
};
