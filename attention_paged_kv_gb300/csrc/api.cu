// The C ABI of the paged-attention library (declared in include/pagedattn.h).
//
// Life cycle as in the FlashInfer issue "How are prefill and decode kernels
// different?": begin_forward (-> pagedattn_plan) once per batch, forward
// (-> pagedattn_run) many times, end_forward (-> pagedattn_plan_destroy).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace {

thread_local std::string g_last_error;

}  // namespace

namespace pa {

pagedattn_status set_err(pagedattn_status s, const std::string& msg) {
  g_last_error = msg;
  return s;
}

pagedattn_status cuda_err(cudaError_t e, const char* what) {
  return set_err(PA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

}  // namespace pa

using pa::cuda_err;
using pa::set_err;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

namespace pa {

// 4-D view of the cache: (D, Hkv, page_size, 2 * num_pages), innermost first.
pagedattn_status encode_kv_map(CUtensorMap* m, const pa::HostPlan& hp, const void* kv, uint32_t box0,
                               uint32_t box2, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_err(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  // NHD: (D, Hkv, ps, 2P); HND: (D, ps, Hkv, 2P) -- innermost first, so a
  // box of rows of one head is {box0, 1, box2, 1} or {box0, box2, 1, 1}
  const cuuint64_t mid1 = hp.hnd ? cuuint64_t(hp.ps) : cuuint64_t(hp.Hkv);
  const cuuint64_t mid2 = hp.hnd ? cuuint64_t(hp.Hkv) : cuuint64_t(hp.ps);
  const cuuint64_t dims[4] = {cuuint64_t(hp.D), mid1, mid2, cuuint64_t(2) * hp.num_pages};
  const cuuint64_t strides[3] = {cuuint64_t(hp.D) * 2, mid1 * hp.D * 2, mid2 * mid1 * hp.D * 2};
  const cuuint32_t box[4] = {box0, hp.hnd ? box2 : 1u, hp.hnd ? 1u : box2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType dt =
      hp.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(m, dt, 4, const_cast<void*>(kv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_err(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed, code " + std::to_string(int(r)));
  return PA_OK;
}

// 3-D view of q: (D, Hq, T), innermost first; box {64, G, 128 / G}: one
// 128-row tile of packed (token, head) rows of one kv head, 128-byte swizzle.
pagedattn_status encode_q_map(CUtensorMap* m, const pa::HostPlan& hp, const void* q, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_err(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {cuuint64_t(hp.D), cuuint64_t(hp.Hq), cuuint64_t(hp.T)};
  const cuuint64_t strides[2] = {cuuint64_t(hp.D) * 2, cuuint64_t(hp.Hq) * hp.D * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(hp.G), cuuint32_t(box_rows / hp.G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      hp.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(m, dt, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_err(PA_ERR_CUDA, "cuTensorMapEncodeTiled (q) failed, code " + std::to_string(int(r)));
  return PA_OK;
}

}  // namespace pa

using pa::encode_kv_map;

namespace {

pagedattn_status fill_inputs(pa::PlanInputs* in, const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                             const int32_t* kv_page_indices, const int32_t* kv_last_page_len, int32_t batch_size,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             int32_t num_pages, pagedattn_dtype dtype, int32_t causal,
                             const pagedattn_options* opts) {
  in->group_indptr = nullptr;
  in->prefix_page_indptr = nullptr;
  in->prefix_page_indices = nullptr;
  in->n_groups = 0;
  in->qo_indptr = qo_indptr;
  in->kv_page_indptr = kv_page_indptr;
  in->kv_page_indices = kv_page_indices;
  in->kv_last_page_len = kv_last_page_len;
  in->B = batch_size;
  in->Hq = num_qo_heads;
  in->Hkv = num_kv_heads;
  in->D = head_dim;
  in->ps = page_size;
  in->num_pages = num_pages;
  in->dtype = int32_t(dtype);
  in->causal = causal ? 1 : 0;
  pagedattn_options o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.reserved[0] != 0) return set_err(PA_ERR_INVALID_ARG, "pagedattn_options.reserved must be zero");
  if (o.wait_limit_cycles < 0) return set_err(PA_ERR_INVALID_ARG, "wait_limit_cycles must be >= 0");
  if (o.kv_layout != PA_LAYOUT_NHD && o.kv_layout != PA_LAYOUT_HND)
    return set_err(PA_ERR_UNSUPPORTED, "kv_layout must be PA_LAYOUT_NHD or PA_LAYOUT_HND");
  if (o.num_sms < 0 || o.decode_chunk_pages < 0 || o.prefill_chunk_tiles < 0)
    return set_err(PA_ERR_INVALID_ARG, "negative option");
  if (o.prefill_q_tiles < 0 || o.prefill_q_tiles > 2)
    return set_err(PA_ERR_INVALID_ARG, "prefill_q_tiles must be 0, 1 or 2");
  if (o.prefill_q_tiles == 2 && head_dim == 256)
    return set_err(PA_ERR_UNSUPPORTED, "head_dim 256 runs one query tile per prefill item");
  in->num_sms = o.num_sms;
  in->force_prefill = o.force_prefill ? 1 : 0;
  in->decode_chunk_pages = o.decode_chunk_pages;
  in->prefill_chunk_tiles = o.prefill_chunk_tiles;
  in->decode_cuda_cores = o.decode_cuda_cores ? 1 : 0;
  in->kv_layout = o.kv_layout;
  in->prefill_q_tiles = o.prefill_q_tiles;
  in->wait_limit_cycles = o.wait_limit_cycles;
  if (in->num_sms == 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || sms < 1) {
      cudaGetLastError();
      return set_err(PA_ERR_INVALID_ARG, "no CUDA device to size the plan for; pass pagedattn_options.num_sms");
    }
    in->num_sms = sms;
  }
  return PA_OK;
}

}  // namespace

namespace pa {

KParams make_params(const RunArgs& a) {
  const HostPlan& hp = *a.hp;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  KParams k;
  std::memset(&k, 0, sizeof(k));
  k.q = a.q;
  k.kv = a.kv;
  k.out = a.out;
  k.lse = a.lse;
  k.pages = reinterpret_cast<const int32_t*>(ws + hp.off_pages);
  k.req = reinterpret_cast<const ReqEntry*>(ws + hp.off_req);
  k.dec = reinterpret_cast<const DecItem*>(ws + hp.off_dec);
  k.pre = reinterpret_cast<const PreItem*>(ws + hp.off_pre);
  k.merge = reinterpret_cast<const MergeEntry*>(ws + hp.off_merge);
  k.part_o = reinterpret_cast<float*>(ws + hp.off_part_o);
  k.part_lse = reinterpret_cast<float*>(ws + hp.off_part_lse);
  k.status = reinterpret_cast<int32_t*>(ws) + H_STATUS;
  k.Hq = hp.Hq;
  k.Hkv = hp.Hkv;
  k.D = hp.D;
  k.ps = hp.ps;
  int s = 0;
  while ((1 << s) < hp.ps) ++s;
  k.ps_shift = s;
  k.G = hp.G;
  s = 0;
  while ((1 << s) < hp.G) ++s;
  k.g_shift = s;
  k.causal = hp.causal;
  k.hnd = hp.hnd;
  k.num_pages = hp.num_pages;
  k.scale_log2 = float(1.4426950408889634 / std::sqrt(double(hp.D)));
  k.wait_limit = hp.wait_limit_cycles > 0 ? (long long)hp.wait_limit_cycles : PA_WAIT_LIMIT_CYCLES;
  k.stall = hp.wait_limit_cycles > 0 ? 1 : 0;
  return k;
}

}  // namespace pa

extern "C" {

const char* pagedattn_version(void) { return "0.2.0"; }

const char* pagedattn_last_error(void) { return g_last_error.c_str(); }

pagedattn_status pagedattn_workspace_size(const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                          const int32_t* kv_page_indices, const int32_t* kv_last_page_len,
                                          int32_t batch_size, int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t page_size, int32_t num_pages,
                                          pagedattn_dtype dtype, int32_t causal, const pagedattn_options* opts,
                                          size_t* bytes) {
  return pagedattn_workspace_size_cascade(nullptr, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len,
                                          batch_size, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages,
                                          dtype, causal, opts, bytes);
}

pagedattn_status pagedattn_workspace_size_cascade(const pagedattn_prefix_groups* groups, const int32_t* qo_indptr,
                                                  const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                                                  const int32_t* kv_last_page_len, int32_t batch_size,
                                                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                                                  int32_t page_size, int32_t num_pages, pagedattn_dtype dtype,
                                                  int32_t causal, const pagedattn_options* opts, size_t* bytes) {
  g_last_error.clear();
  if (!bytes) return set_err(PA_ERR_INVALID_ARG, "bytes is NULL");
  pa::PlanInputs in;
  pagedattn_status s = fill_inputs(&in, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, batch_size,
                                   num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, dtype, causal, opts);
  if (s != PA_OK) return s;
  if (groups) {
    in.group_indptr = groups->group_indptr;
    in.prefix_page_indptr = groups->prefix_page_indptr;
    in.prefix_page_indices = groups->prefix_page_indices;
    in.n_groups = groups->num_groups;
  }
  pa::HostPlan hp;
  std::string err;
  s = pa::build_plan(in, &hp, &err);
  if (s != PA_OK) return set_err(s, err);
  *bytes = hp.total_bytes;
  return PA_OK;
}

pagedattn_status pagedattn_plan(const int32_t* qo_indptr, const int32_t* kv_page_indptr,
                                const int32_t* kv_page_indices, const int32_t* kv_last_page_len, int32_t batch_size,
                                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                int32_t num_pages, pagedattn_dtype dtype, int32_t causal, void* workspace,
                                size_t workspace_bytes, const pagedattn_options* opts, pagedattn_stream_t stream,
                                pagedattn_plan_t* out_plan) {
  return pagedattn_plan_cascade(nullptr, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, batch_size,
                                num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, dtype, causal, workspace,
                                workspace_bytes, opts, stream, out_plan);
}

pagedattn_status pagedattn_plan_cascade(const pagedattn_prefix_groups* groups, const int32_t* qo_indptr,
                                        const int32_t* kv_page_indptr, const int32_t* kv_page_indices,
                                        const int32_t* kv_last_page_len, int32_t batch_size, int32_t num_qo_heads,
                                        int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                        int32_t num_pages, pagedattn_dtype dtype, int32_t causal, void* workspace,
                                        size_t workspace_bytes, const pagedattn_options* opts,
                                        pagedattn_stream_t stream, pagedattn_plan_t* out_plan) {
  g_last_error.clear();
  if (!out_plan) return set_err(PA_ERR_INVALID_ARG, "out_plan is NULL");
  *out_plan = nullptr;
  pa::PlanInputs in;
  pagedattn_status s = fill_inputs(&in, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, batch_size,
                                   num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, dtype, causal, opts);
  if (s != PA_OK) return s;
  if (groups) {
    in.group_indptr = groups->group_indptr;
    in.prefix_page_indptr = groups->prefix_page_indptr;
    in.prefix_page_indices = groups->prefix_page_indices;
    in.n_groups = groups->num_groups;
  }
  pagedattn_plan_s* plan = new pagedattn_plan_s();
  std::string err;
  s = pa::build_plan(in, &plan->hp, &err);
  if (s != PA_OK) {
    delete plan;
    return set_err(s, err);
  }
  plan->force_cp_async = (opts && opts->force_cp_async) ? 1 : 0;
  if (workspace) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256) {
      delete plan;
      return set_err(PA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    }
    if (workspace_bytes < plan->hp.total_bytes) {
      const size_t need = plan->hp.total_bytes;
      delete plan;
      return set_err(PA_ERR_WORKSPACE_TOO_SMALL, "workspace needs " + std::to_string(need) + " bytes, got " +
                                                     std::to_string(workspace_bytes));
    }
    cudaError_t e = cudaGetDevice(&plan->device);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(workspace, plan->hp.blob.data(), plan->hp.blob_bytes, cudaMemcpyHostToDevice,
                          reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      delete plan;
      return cuda_err(e, "plan metadata copy");
    }
    plan->workspace = workspace;
    plan->workspace_bytes = workspace_bytes;
  }
  *out_plan = plan;
  return PA_OK;
}

pagedattn_status pagedattn_run_stages(pagedattn_plan_t plan, const void* q, const void* kv_cache, void* out,
                                      float* lse, pagedattn_stream_t stream, uint32_t stage_mask) {
  if (!plan) return set_err(PA_ERR_INVALID_ARG, "plan is NULL");
  if (!plan->workspace) return set_err(PA_ERR_INVALID_ARG, "host-only plan (built without a workspace)");
  const pa::HostPlan& hp = plan->hp;
  const bool need_rows = hp.T > 0 && (hp.n_pre > 0 || hp.n_dec > 0);
  if (need_rows && (!q || !kv_cache || !out)) return set_err(PA_ERR_INVALID_ARG, "q, kv_cache and out are required");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(out)) %
      16)
    return set_err(PA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
  if (dev != plan->device) return set_err(PA_ERR_INVALID_ARG, "current device differs from the plan's device");
  // make the device's primary context current on this thread: a thread whose
  // first library call is run has none yet, and encoding a tensor map needs one
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_err(e, "cudaSetDevice");

  // the tensor maps of the last pointers seen are cached in the plan; the
  // launches below use copies taken under the plan's lock, so host threads
  // that run one plan at once never see a half-written map
  CUtensorMap map_rows, map_sw128, map_q, map_o[2];
  {
    std::lock_guard<std::mutex> lock(plan->maps_mu);
    if ((hp.n_pre > 0 || hp.n_dec > 0) && kv_cache != plan->map_kv) {
      plan->map_kv = nullptr;
      if (hp.ps >= 8) {
        pagedattn_status s = encode_kv_map(&plan->map_rows, hp, kv_cache, 64, uint32_t(hp.ps < 64 ? hp.ps : 64),
                                           CU_TENSOR_MAP_SWIZZLE_128B);
        if (s != PA_OK) return s;
        s = encode_kv_map(&plan->map_sw128, hp, kv_cache, 64, uint32_t(hp.ps), CU_TENSOR_MAP_SWIZZLE_128B);
        if (s != PA_OK) return s;
      }
      plan->map_kv = kv_cache;
    }
    if (hp.n_pre > 0 && q != plan->map_q_ptr) {
      plan->map_q_ptr = nullptr;
      pagedattn_status s = pa::encode_q_map(&plan->map_q, hp, q);
      if (s != PA_OK) return s;
      plan->map_q_ptr = q;
    }
    if (hp.n_pre > 0 && out != plan->map_o_ptr) {  // full output tiles leave by TMA stores
      plan->map_o_ptr = nullptr;
      pagedattn_status s = pa::encode_q_map(&plan->map_o[0], hp, out);
      if (s == PA_OK) s = pa::encode_q_map(&plan->map_o[1], hp, out, 32);
      if (s != PA_OK) return s;
      plan->map_o_ptr = out;
    }
    map_rows = plan->map_rows;
    map_sw128 = plan->map_sw128;
    map_q = plan->map_q;
    map_o[0] = plan->map_o[0];
    map_o[1] = plan->map_o[1];
  }
  pa::RunArgs a;
  a.hp = &hp;
  a.workspace = plan->workspace;
  a.q = q;
  a.kv = kv_cache;
  a.out = out;
  a.lse = lse;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.force_cp_async = plan->force_cp_async;
  if (stage_mask & PA_STAGE_PREFILL) {
    e = pa::launch_prefill(a, hp.ps >= 8 ? &map_sw128 : nullptr, &map_q, map_o);
    if (e != cudaSuccess) return cuda_err(e, "prefill launch");
  }
  if (stage_mask & PA_STAGE_DECODE) {
    e = pa::launch_decode(a, hp.ps >= 8 ? &map_rows : nullptr);
    if (e != cudaSuccess) return cuda_err(e, "decode launch");
  }
  if (stage_mask & PA_STAGE_MERGE) {
    e = pa::launch_merge(a);
    if (e != cudaSuccess) return cuda_err(e, "merge launch");
  }
  return PA_OK;
}

pagedattn_status pagedattn_run(pagedattn_plan_t plan, const void* q, const void* kv_cache, void* out, float* lse,
                               pagedattn_stream_t stream) {
  return pagedattn_run_stages(plan, q, kv_cache, out, lse, stream, PA_STAGE_ALL);
}

pagedattn_status pagedattn_plan_destroy(pagedattn_plan_t plan) {
  delete plan;
  return PA_OK;
}

pagedattn_status pagedattn_device_status(pagedattn_plan_t plan, pagedattn_stream_t stream, int32_t* flags) {
  if (!plan || !flags) return set_err(PA_ERR_INVALID_ARG, "plan and flags are required");
  if (!plan->workspace) return set_err(PA_ERR_INVALID_ARG, "host-only plan");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t* word = static_cast<int32_t*>(plan->workspace) + pa::H_STATUS;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(word, 0, sizeof(v), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_err(e, "device status read");
  *flags = v;
  if (v & PA_DEV_TIMEOUT) return set_err(PA_ERR_TIMEOUT, "an in-kernel wait gave up after its bound");
  if (v) return set_err(PA_ERR_DEVICE_CHECK, "an in-kernel check fired (flags " + std::to_string(v) + ")");
  return PA_OK;
}

pagedattn_status pagedattn_debug_plan_dump(pagedattn_plan_t plan, void* host_buf, size_t* bytes) {
  if (!plan || !bytes) return set_err(PA_ERR_INVALID_ARG, "plan and bytes are required");
  const size_t n = plan->hp.blob_bytes;
  if (!host_buf) {
    *bytes = n;
    return PA_OK;
  }
  if (*bytes < n) return set_err(PA_ERR_INVALID_ARG, "buffer too small");
  std::memcpy(host_buf, plan->hp.blob.data(), n);
  *bytes = n;
  return PA_OK;
}

pagedattn_status pagedattn_debug_gather(pagedattn_plan_t plan, int32_t* page_out, int32_t* slot_out,
                                        pagedattn_stream_t stream) {
  if (!plan || !page_out || !slot_out) return set_err(PA_ERR_INVALID_ARG, "plan and outputs are required");
  if (!plan->workspace) return set_err(PA_ERR_INVALID_ARG, "host-only plan");
  pa::RunArgs a;
  std::memset(&a, 0, sizeof(a));
  a.hp = &plan->hp;
  a.workspace = plan->workspace;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = pa::launch_debug_gather(a, page_out, slot_out);
  if (e != cudaSuccess) return cuda_err(e, "debug gather launch");
  return PA_OK;
}

}  // extern "C"
