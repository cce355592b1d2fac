// pagedattn_run_decode_noalloc: the decode stages (decode kernel + split
// merge) of a planned batch, for callers that cannot allocate device memory.
//
// Who needs this: serving processes that reserve all free device memory for
// their KV cache up front (a later cudaMalloc fails, or fragments the
// reservation), and latency-critical callers that must not call cudaFree,
// which synchronises the whole device.  Such callers cannot hand the library
// the device workspace that pagedattn_run keeps its metadata and split-KV
// partial states in.  This entry point keeps both in one file-scope device
// array instead, sized kNoallocScratchBytes; it exists once per GPU that
// loads the library and stays allocated until the process exits.
//
// Host code cannot use the array's name as a device address (it is a
// host-side stand-in for the symbol), so the first call on each device looks
// the address up with cudaGetSymbolAddress while that device is current and
// remembers it.  That first call should therefore happen before any stream
// capture.  Every call shares the array: its contents are whatever the last
// call left, each call starts by copying the plan's metadata over it (which
// also clears the status word), and calls that overlap on the GPU (on
// different streams, or from different threads) race on it.  The status word
// the last call's kernels left there is read back by
// pagedattn_noalloc_device_status.
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(16) << 20;  // 16 MiB per GPU
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (which must be current).
pagedattn_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return set_err(PA_ERR_UNSUPPORTED, "device ordinal beyond 63");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return cuda_err(e, "cudaGetSymbolAddress of the no-alloc scratch array");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pagedattn_status pagedattn_run_decode_noalloc(pagedattn_plan_t plan, const void* q,
                                                         const void* kv_cache, void* out, float* lse,
                                                         pagedattn_stream_t stream) {
  using namespace pa;
  if (!plan) return set_err(PA_ERR_INVALID_ARG, "plan is NULL");
  const HostPlan& hp = plan->hp;
  if (hp.n_pre > 0)
    return set_err(PA_ERR_UNSUPPORTED,
                   "pagedattn_run_decode_noalloc runs decode batches only: every request needs qo_len 0 or "
                   "qo_len * G <= 32 with G = num_qo_heads / num_kv_heads in {1, 2, 4, 8, 16}, without "
                   "force_prefill (qo_len 1 and G <= 8 with decode_cuda_cores or at head_dim 256)");
  if (hp.total_bytes > kNoallocScratchBytes)
    return set_err(PA_ERR_WORKSPACE_TOO_SMALL,
                   "this batch needs " + std::to_string(hp.total_bytes) + " bytes of metadata and partial states; "
                   "the no-alloc scratch holds " + std::to_string(kNoallocScratchBytes) +
                   " (plan with a larger decode_chunk_pages, or use pagedattn_run with a workspace)");
  if (hp.n_dec == 0) return PA_OK;
  if (!q || !kv_cache || !out) return set_err(PA_ERR_INVALID_ARG, "q, kv_cache and out are required");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv_cache) | reinterpret_cast<uintptr_t>(out)) %
      16)
    return set_err(PA_ERR_INVALID_ARG, "q, kv_cache and out must be 16-byte aligned");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
  // the device's primary context current on this thread (tensor-map encoding needs one)
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return cuda_err(e, "cudaSetDevice");
  void* scratch = nullptr;
  pagedattn_status s = scratch_address(dev, &scratch);
  if (s != PA_OK) return s;
  CUtensorMap map;
  if (hp.ps >= 8) {
    s = encode_kv_map(&map, hp, kv_cache, 64, uint32_t(hp.ps < 64 ? hp.ps : 64), CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != PA_OK) return s;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // metadata (status word included, as zero) over whatever the last call left
  e = cudaMemcpyAsync(scratch, hp.blob.data(), hp.blob_bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_err(e, "no-alloc metadata copy");
  RunArgs a;
  std::memset(&a, 0, sizeof(a));
  a.hp = &hp;
  a.workspace = scratch;
  a.q = q;
  a.kv = kv_cache;
  a.out = out;
  a.lse = lse;
  a.stream = st;
  e = launch_decode(a, hp.ps >= 8 ? &map : nullptr);
  if (e != cudaSuccess) return cuda_err(e, "no-alloc decode launch");
  e = launch_merge(a);
  if (e != cudaSuccess) return cuda_err(e, "no-alloc merge launch");
  return PA_OK;
}

extern "C" pagedattn_status pagedattn_noalloc_device_status(pagedattn_stream_t stream, int32_t* flags) {
  using namespace pa;
  if (!flags) return set_err(PA_ERR_INVALID_ARG, "flags is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
  void* scratch = nullptr;
  pagedattn_status s = scratch_address(dev, &scratch);
  if (s != PA_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  e = cudaMemcpyAsync(&v, static_cast<int32_t*>(scratch) + H_STATUS, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_err(e, "no-alloc status read");
  *flags = v;
  if (v & PA_DEV_TIMEOUT) return set_err(PA_ERR_TIMEOUT, "an in-kernel wait gave up after its bound");
  if (v) return set_err(PA_ERR_DEVICE_CHECK, "an in-kernel check fired (flags " + std::to_string(v) + ")");
  return PA_OK;
}
