// Shared definitions of the paged-attention library: plan metadata layout,
// kernel parameters, and thin inline-PTX wrappers for the sm_103a features
// the kernels use (mbarrier, TMA tensor copies, cp.async, tcgen05 / TMEM).
//
// Every wait on an mbarrier is bounded: after the run's wait limit (about 2 s
// of clock64 unless the plan set a shorter one), or as soon as another
// thread of the CTA has given up, it returns false and the kernel unwinds
// (see the kernels' abort paths).  Nothing here can spin forever.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/pagedattn.h"
#include "layout.h"

namespace pa {

// Parameters shared by all kernels of one run (passed by value).
struct KParams {
  const void* q;            // [T, Hq, D]
  const void* kv;           // [P, 2, ps, Hkv, D]
  void* out;                // [T, Hq, D]
  float* lse;               // [T, Hq] or nullptr
  const int32_t* pages;     // [nnz] page ids (workspace copy)
  const ReqEntry* req;      // [B]
  const DecItem* dec;       // [n_dec]
  const PreItem* pre;       // [n_pre]
  const MergeEntry* merge;  // [n_merge]
  float* part_o;            // [n_part, D]
  float* part_lse;          // [n_part]
  int32_t* status;          // device status word
  int32_t Hq, Hkv, D, ps, ps_shift, G, g_shift, causal, num_pages, n_items;
  int32_t hnd;              // cache layout: 0 NHD [P, 2, ps, Hkv, D], 1 HND [P, 2, Hkv, ps, D]
  float scale_log2;         // log2(e) / sqrt(D)
  long long wait_limit;     // clock cycles a pipeline wait may poll before it gives up
  int32_t stall;            // test hook: 1 = one thread of every CTA first waits on a barrier
                            // that nothing completes, so that its wait runs out (with a short limit)
};

// ---------------------------------------------------------------------------
// the page-table walk: logical token t of a request -> physical (page, slot)

struct KvLoc { int32_t page; int32_t slot; };

__device__ __forceinline__ KvLoc kv_locate(const int32_t* pages, int32_t page_start, int32_t t,
                                           int32_t ps_shift) {
  KvLoc r;
  r.page = __ldg(pages + page_start + (t >> ps_shift));
  r.slot = t & ((1 << ps_shift) - 1);
  return r;
}

// ---------------------------------------------------------------------------
// small PTX wrappers

// Default bound of a pipeline wait, and the bound of every drain wait (the
// waits that let copies and MMAs in flight land before a CTA exits, which
// never take the shorter limit a caller may set for the pipeline waits).
#ifndef PA_WAIT_LIMIT_CYCLES
#define PA_WAIT_LIMIT_CYCLES (4000000000LL)  // about 2 s at 2 GHz
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Programmatic dependent launch.  Every kernel of a run is launched with
// programmatic stream serialization, so a kernel may start while the kernel
// before it on the stream is still running.  pdl_wait() returns once that
// kernel has completed and its writes are visible; each kernel calls it
// after its prologue (barrier set-up, work-item and page-id reads from the
// plan's metadata, which no kernel writes) and before it reads q, the cache
// or partial states, or writes anything.  pdl_launch() lets the next
// kernel's CTAs be scheduled once every CTA of this grid has issued it (or
// exited); the attention kernels issue it when their main loop is done, so
// the next kernel's prologue overlaps only their epilogue (issued at the
// start, it measured slower on one-wave decode batches).  Launched without
// the attribute, the wait returns at once.  PA_NO_PDL builds without it.
__device__ __forceinline__ void pdl_wait() {
#ifndef PA_NO_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_launch() {
#ifndef PA_NO_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of the same phase (try_wait may suspend the thread for
// a hardware-chosen while before it reports an incomplete phase).
__device__ __forceinline__ bool mbar_test_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Below this many cycles a wait limit polls with non-blocking probes, so that
// the limit and not try_wait's own suspension decides when it gives up.
constexpr long long kShortWaitLimit = 1000000;

// Bounded wait for the phase with the given parity to complete.  Returns
// false (and records PA_DEV_TIMEOUT, and raises *abort_flag) when `limit`
// clock cycles pass or when *abort_flag is already raised by another thread.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status, long long limit) {
  const uint32_t a = smem_u32(bar);
  const bool probe = limit < kShortWaitLimit;
  if (probe ? mbar_test_wait(a, parity) : mbar_try_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (probe ? mbar_test_wait(a, parity) : mbar_try_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, PA_DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Element offset / D of the K (half 0) or V (half 1) row of (page, slot, kv
// head) in the cache, for either layout.
__device__ __forceinline__ size_t kv_row(const KParams& p, int pid, int half, int slot, int h) {
  return p.hnd ? ((size_t(pid) * 2 + half) * p.Hkv + h) * p.ps + slot
               : ((size_t(pid) * 2 + half) * p.ps + slot) * p.Hkv + h;
}

// TMA copy of page rows [slot, slot + box rows) of kv head h, page half z =
// 2 * page + half, columns [c0, c0 + 64), through the 4-D cache map: (D, Hkv,
// ps, 2P) for NHD, (D, ps, Hkv, 2P) for HND.
__device__ __forceinline__ void tma_kv_rows(uint32_t dst, const CUtensorMap* map, int c0, int h, int slot, int z,
                                            uint64_t* bar, int hnd) {
  if (hnd)
    tma_load_4d(dst, map, c0, slot, h, z, bar);
  else
    tma_load_4d(dst, map, c0, h, slot, z, bar);
}

// 3-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled TMA store shared -> global of one box, in the thread's bulk
// group; tma_store_wait_read() returns once every such store of the thread
// has read its shared memory (which may then be reused or released).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(src)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 16-byte cp.async; src_bytes = 0 writes 16 zero bytes without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// tcgen05 / TMEM

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (fp16/bf16 in, fp32 acc).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive fp32 columns; thread i of the warp gets lane
// (lane base + i), columns col..col+31 of the address.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (load).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// 32 lanes x 16 consecutive 32-bit columns (store).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16: A is M rows in TMEM lanes,
// K along columns, two 16-bit elements per 32-bit column.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Wait for this warp's tcgen05.ld; the register pass-through keeps the
// compiler from using the loaded values before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(r[i]));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"): start
// address, leading / stride byte offsets (16-byte units), descriptor
// version 1 at bit 46, swizzle mode in bits 61..63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulate (bits 4-5 = 1), A/B
// element type (bits 7-9 / 10-12: 0 = fp16, 1 = bf16), A and B major-ness
// (bit 15 / 16: 0 = K-major, 1 = MN-major), N >> 3 (bits 17-22), M >> 4
// (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_f16(int ab_bf16, int a_mn_major, int b_mn_major, int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(ab_bf16) << 7) | (static_cast<uint32_t>(ab_bf16) << 10) |
         (static_cast<uint32_t>(a_mn_major) << 15) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// element helpers

template <typename T> struct Elt;
template <> struct Elt<__half> {
  static constexpr int kBf16 = 0;
  __device__ static __forceinline__ float2 to_f2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ static __forceinline__ uint32_t from_f2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ __half from_f(float a) { return __float2half_rn(a); }
};
template <> struct Elt<__nv_bfloat16> {
  static constexpr int kBf16 = 1;
  __device__ static __forceinline__ float2 to_f2(uint32_t w) {
    // bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  __device__ static __forceinline__ uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __device__ static __forceinline__ __nv_bfloat16 from_f(float a) { return __float2bfloat16_rn(a); }
};

}  // namespace pa
