// Decode kernel over the paged KV cache (CUDA cores), the split-KV state
// merge, and the page-walk test kernel.
//
// Decode (one query token per request; "decode kernels use cuda cores", FlashInfer
// issue "How are prefill and decode kernels different?"): one CTA handles one
// work item = (request, kv head, key range).  The key range is a split of the
// request when the planner cut it for kv-parallelism (the issue's split-k);
// a split then writes an fp32 partial state that the merge kernel combines.
//
//   warp 4     producer: TMA copies of whole page rows ([slots, D] of one kv
//              head) through the page table, 64 keys per stage, 3 stages.
//   warps 0-3  each takes 16 of the stage's 64 keys.  A key is read by D/8
//              lanes, 16 bytes each (coalesced rows out of shared memory);
//              every lane holds its 8 columns of q for all G query heads of
//              the group in registers, so each K/V element loaded serves G
//              heads.  Partial dot products are reduce-scattered over the
//              lanes of a key (one shuffle round per halving of the head
//              count), scores go through a small per-warp buffer for the
//              online softmax, and O accumulates in registers.
// At the end the four warps' (max, sum, O) states are combined in shared memory.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kDecThreads = 160;
constexpr int kDecStages = 3;
constexpr int kDecTile = 64;  // keys per stage
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct DecCfg {
  static constexpr int ROW = D * 2;                   // bytes of one K or V row
  static constexpr int STAGE_K = kDecTile * ROW;
  static constexpr int STAGE = 2 * STAGE_K;           // K then V
  static constexpr int OFF_S = kDecStages * STAGE;    // per-warp score buffers
  static constexpr int S_BYTES = 4 * 16 * 8 * 4;      // 4 warps x 16 keys x up to 8 heads
  static constexpr int OFF_BAR = OFF_S + S_BYTES;
  static constexpr int SMEM = OFF_BAR + 128 + 128;
};

template <int N>
struct Log2 { static constexpr int v = 1 + Log2<N / 2>::v; };
template <>
struct Log2<1> { static constexpr int v = 0; };

// Reduce-scatter G per-lane partial sums across the LPT lanes of one key:
// afterwards every lane holds the full sum for head (lane % LPT) / (LPT / G).
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int lane) {
  static_assert(G <= LPT, "group larger than lanes per key");
#pragma unroll
  for (int n = G / 2, off = LPT / 2; n >= 1; n /= 2, off /= 2) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < n; ++k) {
      const float send = upper ? v[k] : v[k + n];
      const float keep = upper ? v[k + n] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float r = v[0];
#pragma unroll
  for (int off = LPT / (2 * G); off >= 1; off /= 2) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const KParams p) {
  using C = DecCfg<D>;
  constexpr int LPT = D / 8;       // lanes per key
  constexpr int TPW = 32 / LPT;    // keys per warp step
  constexpr int STEPS = 16 / TPW;  // steps per warp per stage
  constexpr int VPL = (16 * G >= 32) ? (16 * G) / 32 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + kDecStages;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(empty + kDecStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DecItem it = p.dec[blockIdx.x];
  const ReqEntry rq = p.req[it.req];
  const int nstage = (it.tok1 - it.tok0 + kDecTile - 1) / kDecTile;

  if (tid == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) tma_prefetch_desc(&kv_map);
    const int br_shift = min(p.ps_shift, 6);
    const int BR = 1 << br_shift;  // rows per copy: a page, or 64 slots of it
    int issued = 0;
    for (int j = 0; j < nstage; ++j) {
      const int st = j % kDecStages;
      if (j >= kDecStages) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((j / kDecStages) - 1) & 1, abort_flag, p.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      const int s0 = it.tok0 + j * kDecTile;
      const int s1 = min(s0 + kDecTile, it.tok1);
      const int nbox = (s1 - s0 + BR - 1) >> br_shift;
      if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(nbox * BR * C::ROW * 2));
      __syncwarp();
      const uint32_t kdst = smem_u32(smem) + st * C::STAGE;
      for (int b = lane; b < nbox; b += 32) {
        const KvLoc loc = kv_locate(p.pages, rq.page_start, s0 + b * BR, p.ps_shift);
        int pid = loc.page;
        if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
          atomicOr(p.status, PA_DEV_BAD_INDEX);
          pid = 0;
        }
        tma_load_4d(kdst + b * BR * C::ROW, &kv_map, 0, it.kv_head, loc.slot, 2 * pid, &full[st]);
        tma_load_4d(kdst + C::STAGE_K + b * BR * C::ROW, &kv_map, 0, it.kv_head, loc.slot, 2 * pid + 1, &full[st]);
      }
      issued = j + 1;
    }
    if (lane == 0) {
      for (int j = max(0, issued - kDecStages); j < issued; ++j) {
        const uint32_t a = smem_u32(&full[j % kDecStages]);
        const long long t0 = clock64();
        while (!mbar_try_wait(a, (j / kDecStages) & 1))
          if (clock64() - t0 > PA_WAIT_LIMIT_CYCLES) break;
      }
    }
    __syncwarp();
    asm volatile("bar.arrive 1, 160;" ::: "memory");
    return;
  }

  // ---------------------------------------------------------------- compute warps
  const int tg = lane / LPT;   // key slot within a warp step
  const int ds = lane % LPT;   // 8-column slice
  const int hsel = ds / (LPT / G);
  const bool writer = (ds % (LPT / G)) == 0;
  const int64_t qrow0 = int64_t(rq.qo_start) * p.Hq + int64_t(it.kv_head) * G;

  float qf[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + (qrow0 + g) * D + ds * 8));
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = Elt<T>::to_f2(w4[i]);
      qf[g][2 * i] = f.x * p.scale_log2;
      qf[g][2 * i + 1] = f.y * p.scale_log2;
    }
  }
  float o[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < 8; ++i) o[g][i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;  // state of head (lane % G)
  float* sw = reinterpret_cast<float*>(smem + C::OFF_S) + warp * 16 * G;
  const int hl = lane % G;

  for (int j = 0; j < nstage; ++j) {
    const int st = j % kDecStages;
    bool ok = mbar_wait(&full[st], (j / kDecStages) & 1, abort_flag, p.status);
    if (!__all_sync(0xffffffffu, ok)) break;
    const int s0 = it.tok0 + j * kDecTile;
    const int nval = min(kDecTile, it.tok1 - s0);
    const int wt0 = warp * 16;
    const int wval = max(0, min(16, nval - wt0));
    const uint8_t* kst = smem + st * C::STAGE;
    const uint8_t* vst = kst + C::STAGE_K;

    // scores for this warp's 16 keys
#pragma unroll
    for (int stp = 0; stp < STEPS; ++stp) {
      const int t = stp * TPW + tg;
      const uint4 kraw = *reinterpret_cast<const uint4*>(kst + (wt0 + t) * C::ROW + ds * 16);
      const uint32_t w4[4] = {kraw.x, kraw.y, kraw.z, kraw.w};
      float kf[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = Elt<T>::to_f2(w4[i]);
        kf[2 * i] = f.x;
        kf[2 * i + 1] = f.y;
      }
      float acc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaf(qf[g][i], kf[i], a);
        acc[g] = a;
      }
      const float s = reduce_scatter<G, LPT>(acc, lane);
      if (writer) sw[t * G + hsel] = (t < wval) ? s : -INFINITY;
    }
    __syncwarp();

    // online softmax over the 16 keys, lane owns head hl
    float sv[VPL];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int tt = lane / G + k * (32 / G);
      sv[k] = (tt < 16) ? sw[tt * G + hl] : -INFINITY;
      mx = fmaxf(mx, sv[k]);
    }
#pragma unroll
    for (int off = G; off < 32; off *= 2) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2f(m_run - m_use);
    float psum = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
      const int tt = lane / G + k * (32 / G);
      const float pv = ex2f(sv[k] - m_use);
      if (tt < 16) sw[tt * G + hl] = pv;
      psum += (tt < 16) ? pv : 0.f;
    }
#pragma unroll
    for (int off = G; off < 32; off *= 2) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float ag = __shfl_sync(0xffffffffu, alpha, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[g][i] *= ag;
    }
    __syncwarp();

    // O += P V over the warp's valid keys
#pragma unroll
    for (int stp = 0; stp < STEPS; ++stp) {
      const int t = stp * TPW + tg;
      if (t < wval) {
        const uint4 vraw = *reinterpret_cast<const uint4*>(vst + (wt0 + t) * C::ROW + ds * 16);
        const uint32_t w4[4] = {vraw.x, vraw.y, vraw.z, vraw.w};
        float vf[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = Elt<T>::to_f2(w4[i]);
          vf[2 * i] = f.x;
          vf[2 * i + 1] = f.y;
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pg = sw[t * G + g];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[g][i] = fmaf(pg, vf[i], o[g][i]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // ---------------------------------------------------------------- combine
  // sum O over the TPW key slots of the warp
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int off = LPT; off < 32; off *= 2) o[g][i] += __shfl_xor_sync(0xffffffffu, o[g][i], off);

  // every stage has landed and been read by all four warps: reuse stage memory
  asm volatile("bar.sync 1, 160;" ::: "memory");
  float* comb_o = reinterpret_cast<float*>(smem);       // [4][G][D]
  float* comb_m = comb_o + 4 * G * D;                   // [4][G]
  float* comb_l = comb_m + 4 * G;                       // [4][G]
  if (tg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < 8; ++i) comb_o[(warp * G + g) * D + ds * 8 + i] = o[g][i];
  }
  if (lane < G) {
    comb_m[warp * G + lane] = m_run;
    comb_l[warp * G + lane] = l_run;
  }
  asm volatile("bar.sync 2, 128;" ::: "memory");
  if (*abort_flag) return;

  const bool partial = it.part_row >= 0;
  for (int idx = tid; idx < G * D; idx += 128) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, comb_m[w * G + g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float sc = ex2f(comb_m[w * G + g] - Mu);
      L += sc * comb_l[w * G + g];
      O += sc * comb_o[(w * G + g) * D + d];
    }
    const float val = L > 0.f ? O / L : 0.f;
    const float lse = L > 0.f ? (Mu + __log2f(L)) * kLn2f : -INFINITY;
    if (!partial) {
      static_cast<T*>(p.out)[(qrow0 + g) * D + d] = Elt<T>::from_f(val);
      if (d == 0 && p.lse) p.lse[qrow0 + g] = lse;
    } else {
      p.part_o[(int64_t(it.part_row) + g) * D + d] = val;
      if (d == 0) p.part_lse[it.part_row + g] = lse;
    }
  }
}

// Split-KV merge: one warp per (query token, query head) row of a split
// group.  Each split s holds o_s (already divided by its own softmax sum)
// and lse_s = ln(its sum); the whole sum is sum_s exp(lse_s), so
//   lse = M + ln sum_s exp(lse_s - M),  o = sum_s exp(lse_s - lse) o_s.
template <typename T, int D>
__global__ void __launch_bounds__(256) merge_kernel(const KParams p, const int n_rows) {
  constexpr int V = D / 32;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= n_rows) return;
  const MergeEntry e = p.merge[gw / p.G];
  const int g = gw % p.G;
  float M = -INFINITY;
  for (int s = 0; s < e.nsplit; ++s) M = fmaxf(M, p.part_lse[e.part_row0 + s * e.split_stride + g]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float Z = 0.f;
  for (int s = 0; s < e.nsplit; ++s) {
    const int64_t row = int64_t(e.part_row0) + int64_t(s) * e.split_stride + g;
    const float w = ex2f((p.part_lse[row] - Mu) * kLog2e);
    Z += w;
    const float* src = p.part_o + row * D + lane * V;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = fmaf(w, src[i], acc[i]);
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  const int64_t orow = int64_t(e.out_row0) + g;
  T* dst = static_cast<T*>(p.out) + orow * D + lane * V;
#pragma unroll
  for (int i = 0; i < V; i += 2) {
    const uint32_t w2 = Elt<T>::from_f2(acc[i] * inv, acc[i + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + i) = w2;
  }
  if (lane == 0 && p.lse) p.lse[orow] = Z > 0.f ? Mu + __logf(Z) : -INFINITY;
}

// One block per request: resolve every logical token through the same
// kv_locate the attention kernels use.
__global__ void debug_gather_kernel(const KParams p, const int B, int32_t* page_out, int32_t* slot_out) {
  __shared__ long long off;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    long long s = 0;
    for (int i = 0; i < b; ++i) s += p.req[i].kv_len;
    off = s;
  }
  __syncthreads();
  const ReqEntry rq = p.req[b];
  for (int t = threadIdx.x; t < rq.kv_len; t += blockDim.x) {
    const KvLoc l = kv_locate(p.pages, rq.page_start, t, p.ps_shift);
    page_out[off + t] = l.page;
    slot_out[off + t] = l.slot;
  }
}

template <typename T, int D, int G>
cudaError_t launch_decode_t(const RunArgs& a, const CUtensorMap* map, const KParams& kp) {
  using C = DecCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  decode_kernel<T, D, G><<<a.hp->n_dec, kDecThreads, C::SMEM, a.stream>>>(*map, kp);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_d(const RunArgs& a, const CUtensorMap* map, const KParams& kp) {
  switch (a.hp->G) {
    case 1: return launch_decode_t<T, D, 1>(a, map, kp);
    case 2: return launch_decode_t<T, D, 2>(a, map, kp);
    case 4: return launch_decode_t<T, D, 4>(a, map, kp);
    case 8: return launch_decode_t<T, D, 8>(a, map, kp);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

KParams make_params(const RunArgs& a);

cudaError_t launch_decode(const RunArgs& a, const CUtensorMap* map_rows) {
  if (a.hp->n_dec == 0) return cudaSuccess;
  KParams kp = make_params(a);
  kp.n_items = a.hp->n_dec;
  const bool bf = a.hp->dtype == PA_BF16;
  if (a.hp->D == 128)
    return bf ? launch_decode_d<__nv_bfloat16, 128>(a, map_rows, kp) : launch_decode_d<__half, 128>(a, map_rows, kp);
  return bf ? launch_decode_d<__nv_bfloat16, 64>(a, map_rows, kp) : launch_decode_d<__half, 64>(a, map_rows, kp);
}

cudaError_t launch_merge(const RunArgs& a) {
  if (a.hp->n_merge == 0) return cudaSuccess;
  KParams kp = make_params(a);
  const int rows = a.hp->n_merge * a.hp->G;
  const int blocks = (rows + 7) / 8;
  const bool bf = a.hp->dtype == PA_BF16;
  if (a.hp->D == 128) {
    if (bf) merge_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, a.stream>>>(kp, rows);
    else merge_kernel<__half, 128><<<blocks, 256, 0, a.stream>>>(kp, rows);
  } else {
    if (bf) merge_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, a.stream>>>(kp, rows);
    else merge_kernel<__half, 64><<<blocks, 256, 0, a.stream>>>(kp, rows);
  }
  return cudaGetLastError();
}

cudaError_t launch_debug_gather(const RunArgs& a, int32_t* page_out, int32_t* slot_out) {
  if (a.hp->B == 0) return cudaSuccess;
  KParams kp = make_params(a);
  debug_gather_kernel<<<a.hp->B, 256, 0, a.stream>>>(kp, a.hp->B, page_out, slot_out);
  return cudaGetLastError();
}

}  // namespace pa
