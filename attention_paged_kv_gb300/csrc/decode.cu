// Decode kernel over the paged KV cache (CUDA cores), the split-KV state
// merge, and the page-walk test kernel.
//
// Decode (one query token per request; "decode kernels use cuda cores", FlashInfer
// issue "How are prefill and decode kernels different?"): one CTA handles one
// work item = (request, kv head, key range).  The key range is a split of the
// request when the planner cut it for kv-parallelism (the issue's split-k);
// a split then writes an fp32 partial state that the merge kernel combines.
//
//   warp 4     producer: TMA copies of page rows ([slots, 64 columns] boxes,
//              128-byte swizzle) through the page table, 64 keys per stage,
//              3 stages; pages of fewer than 8 slots go through cp.async with
//              the same swizzle.
//   warps 0..P-1   QK + softmax for P (QK, PV) pairs; warp i takes stages
//              i, i+P, i+2P, ...
//              Each lane owns two keys of the stage and computes their dot
//              products with all G query heads; q (pre-scaled, fp32 column
//              pairs) is read from shared memory by broadcast, K rows through
//              the swizzle without bank conflicts, and no shuffles are needed
//              until the per-head max and sum of the stage.  The warp keeps
//              the running max / sum per head and hands P (and the factor that
//              rescales O) to its PV partner through shared memory.
//   warps P..2P-1  PV: warp P+i accumulates O for warp i's stages; a key's V row
//              is read by D/8 lanes, 16 bytes each, and every lane holds its 8
//              columns of O for all G heads, so one load of a V element feeds
//              G heads.
// The producer is warp 2P.  All products are packed f32x2 FMAs on two
// adjacent head-dim columns.  The pairs keep separate softmax states,
// combined at the end.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

#ifndef PA_DEC_PAIRS
#define PA_DEC_PAIRS 2
#endif
constexpr int kDecPairs = PA_DEC_PAIRS;           // (QK, PV) warp pairs per CTA
constexpr int kDecThreads = 32 * (2 * kDecPairs + 1);  // + 1 producer warp
#ifndef PA_DEC_STAGES
#define PA_DEC_STAGES 3
#endif
constexpr int kDecStages = PA_DEC_STAGES;
constexpr int kDecTile = 64;  // keys per stage
constexpr float kLn2f = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int NST = kDecStages>
struct DecCfg {
  static constexpr int NKB = D / 64;                  // 128-byte column blocks of a row
  static constexpr int BLK = kDecTile * 128;          // 64 rows x 128 bytes
  static constexpr int STAGE_K = NKB * BLK;
  static constexpr int STAGE = 2 * STAGE_K;           // K then V
  static constexpr int OFF_Q = NST * STAGE;          // q: up to 8 heads x D fp32
  static constexpr int OFF_P = OFF_Q + 8 * D * 4;     // P as (p, p) pairs: per pair 64 keys x 8 heads
  static constexpr int OFF_A = OFF_P + kDecPairs * kDecTile * 8 * 8;  // O rescale factor per (pair, head)
  static constexpr int OFF_BAR = OFF_A + kDecPairs * 8 * 4;
  static constexpr int BAR_BYTES = (2 * NST + 2 * kDecPairs) * 8 + 8;  // + abort flag
  static constexpr int OFF_NEVER = OFF_BAR + BAR_BYTES;  // test hook: a barrier nothing completes
  static constexpr int SMEM = OFF_BAR + ((BAR_BYTES + 8 + 127) / 128) * 128 + 1024;  // + alignment slack
};

// Byte offset of 16-byte chunk c (of the row's D/8) of key row t in a stage
// half (K or V) laid out by the 128-byte swizzle: column blocks of 64
// elements, 128-byte rows, chunk index XOR (row mod 8).
template <int D>
__device__ __forceinline__ uint32_t sw_off(int t, int c) {
  return static_cast<uint32_t>((c >> 3) * DecCfg<D>::BLK + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Producer warp of the decode kernels: streams the item's keys in 64-key
// stages (K then V, 128-byte-swizzled rows) into NST buffers, by TMA
// through the page table or, for pages of fewer than 8 slots, by cp.async.
// With TMA it copies the halves [h0, h1) of each stage (0 = K, 1 = V) and
// the 64-column blocks [kb0, kb1) of each row, so several producer warps can
// share a stage's copies; each then arrives on the stage's full barrier with
// its own byte count.  On return every copy it
// issued has landed (or its wait gave up).
template <typename T, int D, int NST = kDecStages>
__device__ __forceinline__ void decode_produce(const CUtensorMap& kv_map, const KParams& p, const DecItem& it,
                                               const ReqEntry& rq, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                               volatile int32_t* abort_flag, int use_tma, int nstage, int lane,
                                               int h0 = 0, int h1 = 2, int kb0 = 0, int kb1 = DecCfg<D>::NKB) {
  using C = DecCfg<D, NST>;
  constexpr int NKB = C::NKB;
  constexpr int NCH = D / 8;
    if (use_tma && lane == 0) tma_prefetch_desc(&kv_map);
    const int br_shift = min(p.ps_shift, 6);
    const int BR = 1 << br_shift;  // rows per copy: a page, or 64 slots of it
    const uint32_t sbase = smem_u32(smem);
    // TMA path: lane b copies box b (a page, or 64 slots of one) of every
    // stage.  Its page id is read three stages ahead into one of three
    // registers (the loop is unrolled by three, so no register of the ring
    // is moved before its load lands), so that no global load sits between
    // a free slot and the copy into it
    auto stage_pid = [&](int jj) -> int {
      if (!use_tma || jj >= nstage) return 0;
      const int s0j = it.tok0 + jj * kDecTile;
      const int nb = (min(s0j + kDecTile, it.tok1) - s0j + BR - 1) >> br_shift;
      return lane < nb ? __ldg(p.pages + it.page_start + ((s0j + lane * BR) >> p.ps_shift)) : 0;
    };
    int pids[3] = {stage_pid(0), stage_pid(1), stage_pid(2)};
    pdl_wait();  // the cache may come from the previous kernel on the stream
    int issued = 0;
    bool ok = true;
    for (int j0 = 0; ok && j0 < nstage; j0 += 3) {
#pragma unroll
     for (int u = 0; u < 3; ++u) {
      const int j = j0 + u;
      if (!ok || j >= nstage) break;
      const int st = j % NST;
      int pid = pids[u];
      pids[u] = stage_pid(j + 3);
      if (j >= NST) {
        if (lane == 0) ok = mbar_wait(&empty[st], ((j / NST) - 1) & 1, abort_flag, p.status, p.wait_limit);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      const int s0 = it.tok0 + j * kDecTile;
      const int s1 = min(s0 + kDecTile, it.tok1);
      const uint32_t kdst = sbase + st * C::STAGE;
      if (use_tma) {
        const int nbox = (s1 - s0 + BR - 1) >> br_shift;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(nbox * BR * 128 * (kb1 - kb0) * (h1 - h0)));
        __syncwarp();
        if (lane < nbox) {
          const int slot = (s0 + lane * BR) & (p.ps - 1);
          if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
            atomicOr(p.status, PA_DEV_BAD_INDEX);
            pid = 0;
          }
#pragma unroll
          for (int kb = 0; kb < NKB; ++kb) {
            if (kb < kb0 || kb >= kb1) continue;
            if (h0 == 0)
              tma_kv_rows(kdst + kb * C::BLK + lane * BR * 128, &kv_map, kb * 64, it.kv_head, slot, 2 * pid,
                          &full[st], p.hnd);
            if (h1 == 2)
              tma_kv_rows(kdst + C::STAGE_K + kb * C::BLK + lane * BR * 128, &kv_map, kb * 64, it.kv_head, slot,
                          2 * pid + 1, &full[st], p.hnd);
          }
        }
      } else {
        const T* kvb = static_cast<const T*>(p.kv);
        for (int t = lane; t < kDecTile; t += 32) {
          const bool valid = s0 + t < s1;
          const T* srck = kvb;
          const T* srcv = kvb;
          if (valid) {
            const KvLoc loc = kv_locate(p.pages, it.page_start, s0 + t, p.ps_shift);
            int pid = loc.page;
            if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.status, PA_DEV_BAD_INDEX);
              pid = 0;
            }
            srck = kvb + kv_row(p, pid, 0, loc.slot, it.kv_head) * D;
            srcv = kvb + kv_row(p, pid, 1, loc.slot, it.kv_head) * D;
          }
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            cp_async16(kdst + sw_off<D>(t, c), srck + (valid ? c * 8 : 0), valid ? 16u : 0u);
            cp_async16(kdst + C::STAGE_K + sw_off<D>(t, c), srcv + (valid ? c * 8 : 0), valid ? 16u : 0u);
          }
        }
        cp_async_commit();
        cp_async_wait_all();
        mbar_arrive(&full[st]);
      }
      issued = j + 1;
     }
    }
    if (use_tma && lane == 0) {
      for (int j = max(0, issued - NST); j < issued; ++j) {
        const uint32_t a = smem_u32(&full[j % NST]);
        const long long t0 = clock64();
        while (!mbar_try_wait(a, (j / NST) & 1))
          if (clock64() - t0 > PA_WAIT_LIMIT_CYCLES) break;
      }
    }
    __syncwarp();
}

template <typename T, int D, int G, int NST>
__global__ void __launch_bounds__(kDecThreads, (NST <= 3 ? 2 : 1))
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const KParams p, const int use_tma) {
  using C = DecCfg<D, NST>;
  constexpr int NKB = C::NKB;
  constexpr int NCH = D / 8;       // 16-byte chunks per row
  constexpr int LPT = D / 8;       // PV lanes per key
  constexpr int TPS = 32 / LPT;    // PV keys per warp step
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NST;
  uint64_t* pfull = empty + NST;  // [pairs] QK -> PV
  uint64_t* pempty = pfull + kDecPairs;  // [pairs] PV -> QK
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(pempty + kDecPairs);
  uint64_t* never = reinterpret_cast<uint64_t*>(smem + C::OFF_NEVER);
  float2* qs2 = reinterpret_cast<float2*>(smem + C::OFF_Q);  // [G][D/2]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DecItem it = p.dec[blockIdx.x];
  const ReqEntry rq = p.req[it.req];
  const int nstage = (it.tok1 - it.tok0 + kDecTile - 1) / kDecTile;
  const int64_t qrow0 = int64_t(rq.qo_start) * p.Hq + int64_t(it.kv_head) * G;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], use_tma ? 1 : 32);
      mbar_init(&empty[i], 2);
    }
    for (int i = 0; i < kDecPairs; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], 1);
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  pdl_wait();  // q may come from the previous kernel on the stream
  // q for the G heads, pre-scaled into log2 units, as fp32 column pairs
  for (int idx = tid; idx < G * D / 2; idx += kDecThreads) {
    const int g = idx / (D / 2), c2 = idx % (D / 2);
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const T*>(p.q) + (qrow0 + g) * D) + c2);
    qs2[idx] = __fmul2_rn(Elt<T>::to_f2(w), make_float2(p.scale_log2, p.scale_log2));
  }
  __syncthreads();

  if (p.stall && warp == 0) mbar_wait(never, 0, abort_flag, p.status, p.wait_limit);  // test hook
  if (warp == 2 * kDecPairs) {
    decode_produce<T, D, NST>(kv_map, p, it, rq, smem, full, empty, abort_flag, use_tma, nstage, lane);
    asm volatile("bar.arrive 1, %0;" ::"n"(kDecThreads) : "memory");
    return;
  }

  const int pair = warp % kDecPairs;
  float2* pbuf = reinterpret_cast<float2*>(smem + C::OFF_P) + pair * kDecTile * 8;  // [64 keys][8 heads]
  float* abuf = reinterpret_cast<float*>(smem + C::OFF_A) + pair * 8;
  float* comb_o = reinterpret_cast<float*>(smem);  // [pairs][G][D], reuses stage memory at the end
  float* comb_m = comb_o + kDecPairs * G * D;      // [pairs][G]
  float* comb_l = comb_m + kDecPairs * G;          // [pairs][G]

  if (warp < kDecPairs) {
    // ---------------------------------------------------------------- QK + softmax
    float m_run[G], l_run[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
    }
    const int t0 = lane, t1 = lane + 32;
    for (int k = 0, j = pair; j < nstage; ++k, j += kDecPairs) {
      const int st = j % NST;
      bool ok = mbar_wait(&full[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int nval = min(kDecTile, it.tok1 - (it.tok0 + j * kDecTile));
      const uint8_t* kst = smem + st * C::STAGE;
      float2 a0[G], a1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        a0[g] = make_float2(0.f, 0.f);
        a1[g] = make_float2(0.f, 0.f);
      }
#pragma unroll 4
      for (int c = 0; c < NCH; ++c) {
        const uint4 r0 = *reinterpret_cast<const uint4*>(kst + sw_off<D>(t0, c));
        const uint4 r1 = *reinterpret_cast<const uint4*>(kst + sw_off<D>(t1, c));
        const float2 k0[4] = {Elt<T>::to_f2(r0.x), Elt<T>::to_f2(r0.y), Elt<T>::to_f2(r0.z), Elt<T>::to_f2(r0.w)};
        const float2 k1[4] = {Elt<T>::to_f2(r1.x), Elt<T>::to_f2(r1.y), Elt<T>::to_f2(r1.z), Elt<T>::to_f2(r1.w)};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(qs2 + g * (D / 2) + c * 4);
          const float4 qb = *reinterpret_cast<const float4*>(qs2 + g * (D / 2) + c * 4 + 2);
          const float2 q4[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w), make_float2(qb.x, qb.y),
                                make_float2(qb.z, qb.w)};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a0[g] = __ffma2_rn(q4[i], k0[i], a0[g]);
            a1[g] = __ffma2_rn(q4[i], k1[i], a1[g]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with K of the stage

      float alpha[G], p0[G], p1[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float s0 = (t0 < nval) ? a0[g].x + a0[g].y : -INFINITY;
        const float s1 = (t1 < nval) ? a1[g].x + a1[g].y : -INFINITY;
        float mx = fmaxf(s0, s1);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m_run[g], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[g] = ex2f(m_run[g] - m_use);
        p0[g] = ex2f(s0 - m_use);
        p1[g] = ex2f(s1 - m_use);
        float sum = p0[g] + p1[g];
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        l_run[g] = l_run[g] * alpha[g] + sum;
        m_run[g] = m_new;
      }
      if (k >= 1) {
        ok = mbar_wait(&pempty[pair], (k - 1) & 1, abort_flag, p.status, p.wait_limit);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pbuf[t0 * 8 + g] = make_float2(p0[g], p0[g]);
        pbuf[t1 * 8 + g] = make_float2(p1[g], p1[g]);
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) abuf[g] = alpha[g];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[pair]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory");
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        comb_m[pair * G + g] = m_run[g];
        comb_l[pair * G + g] = l_run[g];
      }
    }
  } else {
    // ---------------------------------------------------------------- PV
    const int tg = lane / LPT;  // key slot within a warp step
    const int ds = lane % LPT;  // 8-column slice
    float2 o2[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i) o2[g][i] = make_float2(0.f, 0.f);
    for (int k = 0, j = pair; j < nstage; ++k, j += kDecPairs) {
      const int st = j % NST;
      bool ok = mbar_wait(&full[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
      if (ok) ok = mbar_wait(&pfull[pair], k & 1, abort_flag, p.status, p.wait_limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int nval = min(kDecTile, it.tok1 - (it.tok0 + j * kDecTile));
      const uint8_t* vst = smem + st * C::STAGE + C::STAGE_K;
      bool resc = false;
      float al[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        al[g] = abuf[g];
        resc |= (al[g] != 1.f);
      }
      if (resc) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < 4; ++i) o2[g][i] = __fmul2_rn(o2[g][i], make_float2(al[g], al[g]));
      }
#pragma unroll 4
      for (int t = tg; t < nval; t += TPS) {
        const uint4 vr = *reinterpret_cast<const uint4*>(vst + sw_off<D>(t, ds));
        const float2 v2[4] = {Elt<T>::to_f2(vr.x), Elt<T>::to_f2(vr.y), Elt<T>::to_f2(vr.z), Elt<T>::to_f2(vr.w)};
        float2 pp[G];
#pragma unroll
        for (int g = 0; g < G; g += 2) {
          const float4 pv = *reinterpret_cast<const float4*>(pbuf + t * 8 + g);
          pp[g] = make_float2(pv.x, pv.y);
          if (g + 1 < G) pp[g + 1] = make_float2(pv.z, pv.w);
        }
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int i = 0; i < 4; ++i) o2[g][i] = __ffma2_rn(pp[g], v2[i], o2[g][i]);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&pempty[pair]);
        mbar_arrive(&empty[st]);
      }
    }
    // sum O over the TPS key slots of the warp
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int off = LPT; off < 32; off *= 2) {
          o2[g][i].x += __shfl_xor_sync(0xffffffffu, o2[g][i].x, off);
          o2[g][i].y += __shfl_xor_sync(0xffffffffu, o2[g][i].y, off);
        }
    // every stage has landed and been read: stage memory can be reused
    asm volatile("bar.sync 1, %0;" ::"n"(kDecThreads) : "memory");
    if (tg == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float2*>(&comb_o[(pair * G + g) * D + ds * 8 + 2 * i]) = o2[g][i];
    }
  }

  pdl_launch();
  // ---------------------------------------------------------------- combine the pairs
  asm volatile("bar.sync 2, %0;" ::"n"(64 * kDecPairs) : "memory");
  if (*abort_flag) return;
  const bool partial = it.part_row >= 0;
  for (int idx = tid; idx < G * D; idx += 64 * kDecPairs) {
    const int g = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kDecPairs; ++q) M = fmaxf(M, comb_m[q * G + g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int q = 0; q < kDecPairs; ++q) {
      const float wq = ex2f(comb_m[q * G + g] - Mu);
      L += wq * comb_l[q * G + g];
      O += wq * comb_o[(q * G + g) * D + d];
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

// ---------------------------------------------------------------------------
// Small-query kernel on the tensor cores (warp-level MMA, m16n8k16, fp32
// accumulate): decode, and requests of a few query tokens (speculative
// decoding, small chunks) whose qo_len * G packed (token, head) rows number
// at most 32.  Launches of no more CTAs than SMs run one CTA per SM with six
// 64-key stages (192 KB in flight); larger ones two CTAs per SM with three.
//
// At G query heads per kv head the CUDA-core kernel above needs 2*G MACs per
// cached element, more than the FP32 pipe sustains at HBM speed once G >= 4;
// the FlashInfer issue "How are prefill and decode kernels different?" makes
// the same point (tensor cores pay off for grouped-query decode) and names a
// small-query variant of the prefill kernel as missing.  Here the packed rows
// r = token * G + head of an item are the M rows of m16n8k16 fragments, so
// S = q K^T needs no reshaping:
//   warps 4-5  the producer of the CUDA-core kernel (64-key stages, 128-byte
//   (or 4-7)   swizzled rows), split in two: warp 4 copies the stages' K,
//              warp 5 their V (each TMA copy costs its issuing warp ~110
//              cycles, and one warp issuing all copies limited a CTA's
//              stream: mixed-batch decode 0.712 -> 0.698 ms).  Launches of
//              one CTA per SM at head_dim 128 split each half again by
//              64-column block over four warps (two warps' issue time still
//              set the pace there: decode timing script 14.6 -> 13.9 us).
//              With cp.async staging warp 4 copies everything.
//   warps 0-3  row group rg = warp % RGN (16 rows each), key subset
//              kq = warp / RGN of every stage: with RGN row groups each warp
//              takes 16 * RGN of the stage's 64 keys.  ldmatrix feeds K from
//              the swizzled rows; the online softmax runs on the accumulator
//              fragment (a quad of lanes holds a row), whose exp2 values
//              become the A fragment of P V directly; ldmatrix.trans feeds V.
//              O stays in registers; the key subsets are combined at the end.
// Row classes (template RC): up to 8 rows, up to 16 (RGN 1; fragment rows
// past R see no keys) and 32 (RGN 2).  Class 0 (up to 8 rows) computes the
// transposed products instead (S^T = K q^T, O^T = V^T P^T: the rows on the
// MMAs' 8-wide N side, half the MMAs of the direct form, which leaves 8 of
// 16 M rows idle).  (64 rows, RGN 4, is never planned: there the warp-level
// MMA bound the kernel at 43 % of HBM, and the tcgen05 prefill kernel is
// faster.)  Each row's keys end at its own causal limit.  For requests with
// fewer than 128 keys P is split into hi + lo halves (two MMAs), as in the
// prefill kernel, so rows that see few keys keep P's rounding out of the
// output.

template <typename T>
struct Mma {
  // all 16 rows; a = {row g cols 2t.., row g cols 2t+8.., row g+8 cols 2t.., row g+8 cols 2t+8..}
  __device__ static __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (Elt<T>::kBf16)
      asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
          : "r"(a[0]), "r"(a[2]), "r"(a[1]), "r"(a[3]), "r"(b0), "r"(b1));
    else
      asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
          "{%0, %1, %2, %3};"
          : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
          : "r"(a[0]), "r"(a[2]), "r"(a[1]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}
// 8x8 transpose of 16-bit elements across the warp: lane (g, t) holds
// elements (g, 2t) and (g, 2t + 1) before and after
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Producer warps of the small-query kernel: two (K, V) when two CTAs share
// an SM; four (K and V of each 64-column block) in the one-CTA-per-SM
// launches at head_dim 128, where each producer warp's issue time (about
// 110 cycles a copy, 8 copies of a stage for one warp) set the pace.
template <int D, int NST>
__host__ __device__ constexpr int dm_prods() { return (NST > kDecStages && D >= 128) ? 4 : 2; }
template <int D, int NST>
__host__ __device__ constexpr int dm_threads() { return 32 * (4 + dm_prods<D, NST>()); }

template <int RC>
struct RowClass {
  static_assert(RC >= 0 && RC <= 2, "row classes of up to 32 rows");
  static constexpr int RGN = RC <= 1 ? 1 : 2;                  // row groups of 16
  static constexpr int KS = 4 / RGN;                           // key subsets (warps per row group)
  static constexpr int KW = kDecTile / KS;                     // keys per warp per stage
  static constexpr int NKB = KW / 16;                          // 16-key blocks per warp
};

template <typename T, int D, int RC, int NST>
__global__ void __launch_bounds__(dm_threads<D, NST>(), NST <= 3 ? 2 : 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap kv_map, const KParams p, const int use_tma,
                      const int item0) {
  using C = DecCfg<D, NST>;
  using RCl = RowClass<RC>;
  constexpr int PRODS = dm_prods<D, NST>(), THREADS = dm_threads<D, NST>();
  constexpr int RGN = RCl::RGN, KS = RCl::KS, KW = RCl::KW, NKB = RCl::NKB;
  constexpr int NA = 4;        // fragment registers per lane: rows lo (0, 1) and hi (2, 3)
  constexpr int NKS = D / 16;  // k-steps of S
  constexpr int NNT = D / 8;   // n-tiles of O
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + NST;
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(empty + NST);
  uint64_t* never = reinterpret_cast<uint64_t*>(smem + C::OFF_NEVER);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DecItem it = p.dec[item0 + blockIdx.x];
  const ReqEntry rq = p.req[it.req];
  const int nstage = (it.tok1 - it.tok0 + kDecTile - 1) / kDecTile;
  const int R = rq.qo_len << p.g_shift;  // packed rows: r = token * G + head

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], use_tma ? PRODS : 32);
      mbar_init(&empty[i], 4);
    }
    mbar_init(never, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp >= 4) {
    // with TMA staging producer warp 4 + w copies half w % 2 (K, V) of every
    // stage, and with four producers column block w / 2 of it; cp.async
    // staging (pages of < 8 slots) stays with warp 4 alone
    if (warp == 4 || use_tma) {
      const int w = warp - 4;
      const int h0 = use_tma ? (w & 1) : 0, h1 = use_tma ? (w & 1) + 1 : 2;
      const int kb0 = (use_tma && PRODS == 4) ? (w >> 1) : 0;
      const int kb1 = (use_tma && PRODS == 4) ? (w >> 1) + 1 : C::NKB;
      decode_produce<T, D, NST>(kv_map, p, it, rq, smem, full, empty, abort_flag, use_tma, nstage, lane, h0, h1,
                                kb0, kb1);
    }
    asm volatile("bar.arrive 1, %0;" ::"n"(THREADS) : "memory");
    return;
  }

  if (p.stall && warp == 0) mbar_wait(never, 0, abort_flag, p.status, p.wait_limit);  // test hook
  pdl_wait();  // q may come from the previous kernel on the stream
  const int rg = warp % RGN, kq = warp / RGN;
  const int g = lane >> 2, t = lane & 3;    // fragment row and column pair
  const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row this lane addresses
  const int r_lo = rg * 16 + g, r_hi = r_lo + 8;
  // global q / out row of packed row r
  auto row_of = [&](int r) -> int64_t {
    return int64_t(rq.qo_start + (r >> p.g_shift)) * p.Hq + int64_t(it.kv_head) * p.G + (r & (p.G - 1));
  };
  // end (exclusive, absolute key position) of the keys row r may see in this item:
  // the item's range, cut at the row's bottom-right causal limit
  auto end_of = [&](int r) -> int {
    if (r >= R) return 0;
    const int lim = p.causal ? rq.kv_len - rq.qo_len + (r >> p.g_shift) + 1 : rq.kv_len;
    return min(it.tok1, lim);
  };
  const int end_lo = end_of(r_lo), end_hi = end_of(r_hi);
  float* comb_o = reinterpret_cast<float*>(smem);  // [4 warps][16 rows][D], over the stages at the end
  float* comb_m = comb_o + 4 * 16 * D;             // [4][16]
  float* comb_l = comb_m + 4 * 16;                 // [4][16]

  if constexpr (RC == 0) {
    // Up to 8 packed rows: S^T = K q^T and O^T = V^T P^T, so the 16-row (M)
    // side of each m16n8k16 holds keys or head-dim columns and its 8-column
    // (N) side the packed rows: no MMA row idles (the direct form below
    // fills 8 of its 16 rows, twice the MMAs a stage).  Warp w takes keys
    // 16w .. 16w + 15 of every stage; lane (g, t) holds S^T of keys g and
    // g + 8 for rows 2t and 2t + 1, and O^T of columns g and g + 8 of each
    // 16-column block for the same two rows.  P^T reaches the B operand of
    // O^T through 8x8 transposes in registers.
    constexpr int NMT = D / 16;  // 16-column blocks of O^T
    const int kofs = warp * 16;
    const int ra = 2 * t, rb = 2 * t + 1;
    const int end_a = end_of(ra), end_b = end_of(rb);
    // q^T as B fragments: {q[row g][16 kk + 2t ..], q[row g][16 kk + 2t + 8 ..]}
    uint32_t qb[NKS][2];
#pragma unroll
    for (int kk = 0; kk < NKS; ++kk) qb[kk][0] = qb[kk][1] = 0u;
    if (g < R) {
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(static_cast<const T*>(p.q) + row_of(g) * D);
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk) {
        qb[kk][0] = __ldg(qp + kk * 8 + t);
        qb[kk][1] = __ldg(qp + kk * 8 + 4 + t);
      }
    }
    float ot[NMT][4];  // {col 16m + g: rows a, b; col 16m + g + 8: rows a, b}
#pragma unroll
    for (int m = 0; m < NMT; ++m)
#pragma unroll
      for (int e = 0; e < 4; ++e) ot[m][e] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY;
    float l_a = 0.f, l_b = 0.f;  // sums over this lane's keys only
    const bool split_p = rq.kv_len < 128;
    const float sl2 = p.scale_log2;
    for (int j = 0; j < nstage; ++j) {
      const int st = j % NST;
      const bool ok = mbar_wait(&full[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int s0 = it.tok0 + j * kDecTile;
      const int nval = min(kDecTile, it.tok1 - s0);
      const uint32_t kbase = smem_u32(smem) + st * C::STAGE;
      const uint32_t vbase = kbase + C::STAGE_K;
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk) {
        uint32_t a[4];
        ldsm_x4(kbase + sw_off<D>(kofs + (mi >> 1) * 8 + ri, 2 * kk + (mi & 1)), a[0], a[1], a[2], a[3]);
        Mma<T>::run(sc, a, qb[kk][0], qb[kk][1]);
      }
      // each row's keys end at its own causal limit
      const int key0 = s0 + kofs + g, key1 = key0 + 8;
      sc[0] = key0 < end_a ? sc[0] * sl2 : -INFINITY;
      sc[1] = key0 < end_b ? sc[1] * sl2 : -INFINITY;
      sc[2] = key1 < end_a ? sc[2] * sl2 : -INFINITY;
      sc[3] = key1 < end_b ? sc[3] * sl2 : -INFINITY;
      float mx_a = fmaxf(sc[0], sc[2]), mx_b = fmaxf(sc[1], sc[3]);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, sh));
        mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, sh));
      }
      // a row that has seen no key yet keeps O = 0 and needs no rescale
      const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
      const float mu_a = (mn_a == -INFINITY) ? 0.f : mn_a;
      const float mu_b = (mn_b == -INFINITY) ? 0.f : mn_b;
      const float al_a = (mn_a == -INFINITY) ? 1.f : ex2f(m_a - mu_a);
      const float al_b = (mn_b == -INFINITY) ? 1.f : ex2f(m_b - mu_b);
      m_a = mn_a;
      m_b = mn_b;
      const float p0 = ex2f(sc[0] - mu_a), p1 = ex2f(sc[1] - mu_b);
      const float p2 = ex2f(sc[2] - mu_a), p3 = ex2f(sc[3] - mu_b);
      l_a = l_a * al_a + (p0 + p2);
      l_b = l_b * al_b + (p1 + p3);
      if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
        for (int m = 0; m < NMT; ++m) {
          ot[m][0] *= al_a;
          ot[m][1] *= al_b;
          ot[m][2] *= al_a;
          ot[m][3] *= al_b;
        }
      }
      // P^T as B fragments ({keys 2t, 2t + 1 | row g}, {keys 2t + 8, 2t + 9 |
      // row g}), plus the rounding remainder when P is split
      const uint32_t x0 = Elt<T>::from_f2(p0, p1), x1 = Elt<T>::from_f2(p2, p3);
      const uint32_t pb0 = movm_t(x0), pb1 = movm_t(x1);
      uint32_t lb0 = 0u, lb1 = 0u;
      if (split_p) {
        const float2 h0 = Elt<T>::to_f2(x0), h1 = Elt<T>::to_f2(x1);
        lb0 = movm_t(Elt<T>::from_f2(p0 - h0.x, p1 - h0.y));
        lb1 = movm_t(Elt<T>::from_f2(p2 - h1.x, p3 - h1.y));
      }
      // O^T += V^T P^T; V rows past the range (other data, or stale stage
      // contents: possibly NaN) are zeroed in the fragments
      uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
      if (nval < kofs + 16) {
        const int k0 = kofs + 2 * t;  // ldmatrix.trans: this lane's keys 2t, 2t + 1 (+ 8)
        mlo = (k0 < nval ? 0x0000ffffu : 0u) | (k0 + 1 < nval ? 0xffff0000u : 0u);
        mhi = (k0 + 8 < nval ? 0x0000ffffu : 0u) | (k0 + 9 < nval ? 0xffff0000u : 0u);
      }
#pragma unroll
      for (int m = 0; m < NMT; ++m) {
        uint32_t a[4];
        ldsm_x4_t(vbase + sw_off<D>(kofs + (mi & 1) * 8 + ri, 2 * m + (mi >> 1)), a[0], a[1], a[2], a[3]);
        a[0] &= mlo;
        a[1] &= mhi;
        a[2] &= mlo;
        a[3] &= mhi;
        Mma<T>::run(ot[m], a, pb0, pb1);
        if (split_p) Mma<T>::run(ot[m], a, lb0, lb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    pdl_launch();
    // ---------------------------------------------------------------- combine the key subsets
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
      l_a += __shfl_xor_sync(0xffffffffu, l_a, sh);
      l_b += __shfl_xor_sync(0xffffffffu, l_b, sh);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");  // stage memory is free from here
#pragma unroll
    for (int m = 0; m < NMT; ++m) {
      comb_o[(warp * 16 + ra) * D + 16 * m + g] = ot[m][0];
      comb_o[(warp * 16 + rb) * D + 16 * m + g] = ot[m][1];
      comb_o[(warp * 16 + ra) * D + 16 * m + g + 8] = ot[m][2];
      comb_o[(warp * 16 + rb) * D + 16 * m + g + 8] = ot[m][3];
    }
    if (g == 0) {
      comb_m[warp * 16 + ra] = m_a;
      comb_l[warp * 16 + ra] = l_a;
      comb_m[warp * 16 + rb] = m_b;
      comb_l[warp * 16 + rb] = l_b;
    }
  } else {

    // q as A fragments: {row lo cols 2t, row lo cols 2t+8, row hi cols 2t, row hi cols 2t+8} per k-step
    uint32_t qa[NKS][NA];
    {
      const T* q = static_cast<const T*>(p.q);
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk) qa[kk][0] = qa[kk][1] = 0u;
      if (r_lo < R) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(q + row_of(r_lo) * D);
#pragma unroll
        for (int kk = 0; kk < NKS; ++kk) {
          qa[kk][0] = __ldg(qp + kk * 8 + t);
          qa[kk][1] = __ldg(qp + kk * 8 + 4 + t);
        }
      }
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk) qa[kk][2] = qa[kk][3] = 0u;
      if (r_hi < R) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(q + row_of(r_hi) * D);
#pragma unroll
        for (int kk = 0; kk < NKS; ++kk) {
          qa[kk][2] = __ldg(qp + kk * 8 + t);
          qa[kk][3] = __ldg(qp + kk * 8 + 4 + t);
        }
      }
    }
    float o[NNT][NA];  // rows lo (regs 0, 1) and hi (2, 3); columns 8n + 2t, 8n + 2t + 1
#pragma unroll
    for (int n = 0; n < NNT; ++n)
#pragma unroll
      for (int e = 0; e < NA; ++e) o[n][e] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY;
    float l_lo = 0.f, l_hi = 0.f;  // sums over this lane's columns only
    const bool split_p = rq.kv_len < 128;
    const float sl2 = p.scale_log2;
    const int kofs = kq * KW;  // this warp's first key in every stage

    for (int j = 0; j < nstage; ++j) {
      const int st = j % NST;
      const bool ok = mbar_wait(&full[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
      if (!__all_sync(0xffffffffu, ok)) break;
      const int s0 = it.tok0 + j * kDecTile;         // absolute position of the stage's first key
      const int nval = min(kDecTile, it.tok1 - s0);  // keys of the stage inside the item's range
      const uint32_t kbase = smem_u32(smem) + st * C::STAGE;
      const uint32_t vbase = kbase + C::STAGE_K;

      // S = q K^T for keys kofs .. kofs + KW - 1 of the stage (n-tiles of 8 keys)
      float sc[2 * NKB][NA];
#pragma unroll
      for (int n = 0; n < 2 * NKB; ++n)
#pragma unroll
        for (int e = 0; e < NA; ++e) sc[n][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < NKS; ++kk) {
#pragma unroll
        for (int kb = 0; kb < NKB; ++kb) {
          uint32_t b00, b01, b10, b11;
          ldsm_x4(kbase + sw_off<D>(kofs + kb * 16 + (mi >> 1) * 8 + ri, 2 * kk + (mi & 1)), b00, b01, b10, b11);
          Mma<T>::run(sc[2 * kb], qa[kk], b00, b01);
          Mma<T>::run(sc[2 * kb + 1], qa[kk], b10, b11);
        }
      }

      // online softmax on the fragment: this lane holds keys 8n + 2t + e of rows lo and hi
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2 * NKB; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = s0 + kofs + n * 8 + 2 * t + e;
          sc[n][e] = key < end_lo ? sc[n][e] * sl2 : -INFINITY;
          mx_lo = fmaxf(mx_lo, sc[n][e]);
          sc[n][2 + e] = key < end_hi ? sc[n][2 + e] * sl2 : -INFINITY;
          mx_hi = fmaxf(mx_hi, sc[n][2 + e]);
        }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      // a row that has seen no key yet keeps O = 0 and needs no rescale (alpha 1)
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float mu_lo = (mn_lo == -INFINITY) ? 0.f : mn_lo;
      const float mu_hi = (mn_hi == -INFINITY) ? 0.f : mn_hi;
      const float al_lo = (mn_lo == -INFINITY) ? 1.f : ex2f(m_lo - mu_lo);
      const float al_hi = (mn_hi == -INFINITY) ? 1.f : ex2f(m_hi - mu_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float ps_lo = 0.f, ps_hi = 0.f;
#pragma unroll
      for (int n = 0; n < 2 * NKB; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[n][e] = ex2f(sc[n][e] - mu_lo);
          ps_lo += sc[n][e];
          sc[n][2 + e] = ex2f(sc[n][2 + e] - mu_hi);
          ps_hi += sc[n][2 + e];
        }
      l_lo = l_lo * al_lo + ps_lo;
      l_hi = l_hi * al_hi + ps_hi;
      if (__any_sync(0xffffffffu, al_lo != 1.f || al_hi != 1.f)) {
#pragma unroll
        for (int n = 0; n < NNT; ++n) {
          o[n][0] *= al_lo;
          o[n][1] *= al_lo;
          o[n][2] *= al_hi;
          o[n][3] *= al_hi;
        }
      }

      // P as A fragments of P V, one per 16-key block (n-tiles 2kb, 2kb + 1),
      // plus the rounding remainder when P is split
      uint32_t pa[NKB][NA], la[NKB][NA];
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int x = 0; x < NA; ++x) {
          // x = 0, 1: row lo, keys 2t.. and 8 + 2t..; x = 2, 3: row hi
          const float v0 = sc[2 * kb + (x & 1)][(x >> 1) * 2];
          const float v1 = sc[2 * kb + (x & 1)][(x >> 1) * 2 + 1];
          pa[kb][x] = Elt<T>::from_f2(v0, v1);
          la[kb][x] = 0u;
          if (split_p) {
            const float2 h = Elt<T>::to_f2(pa[kb][x]);
            la[kb][x] = Elt<T>::from_f2(v0 - h.x, v1 - h.y);
          }
        }

      // O += P V; V rows of keys past the range (other data, or stale stage
      // contents: possibly NaN) are zeroed in the fragments, since 0 * NaN = NaN
      const bool vpart = nval < kofs + KW;
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (vpart) {
          const int k0 = kofs + kb * 16 + 2 * t;  // ldmatrix.trans: this lane's keys 2t, 2t+1 (+8)
          mlo = (k0 < nval ? 0x0000ffffu : 0u) | (k0 + 1 < nval ? 0xffff0000u : 0u);
          mhi = (k0 + 8 < nval ? 0x0000ffffu : 0u) | (k0 + 9 < nval ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int dp = 0; dp < NNT / 2; ++dp) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(vbase + sw_off<D>(kofs + kb * 16 + (mi & 1) * 8 + ri, 2 * dp + (mi >> 1)), v0, v1, v2, v3);
          v0 &= mlo;
          v1 &= mhi;
          v2 &= mlo;
          v3 &= mhi;
          Mma<T>::run(o[2 * dp], pa[kb], v0, v1);
          Mma<T>::run(o[2 * dp + 1], pa[kb], v2, v3);
          if (split_p) {
            Mma<T>::run(o[2 * dp], la[kb], v0, v1);
            Mma<T>::run(o[2 * dp + 1], la[kb], v2, v3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    pdl_launch();
    // ---------------------------------------------------------------- combine the key subsets
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");  // stage memory is free from here
#pragma unroll
    for (int n = 0; n < NNT; ++n) {
      *reinterpret_cast<float2*>(&comb_o[(warp * 16 + g) * D + n * 8 + 2 * t]) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(&comb_o[(warp * 16 + g + 8) * D + n * 8 + 2 * t]) = make_float2(o[n][2], o[n][3]);
    }
    if (t == 0) {
      comb_m[warp * 16 + g] = m_lo;
      comb_l[warp * 16 + g] = l_lo;
      comb_m[warp * 16 + g + 8] = m_hi;
      comb_l[warp * 16 + g + 8] = l_hi;
    }
  }
  asm volatile("bar.sync 2, 128;" ::: "memory");
  if (*abort_flag) return;
  const bool partial = it.part_row >= 0;
  // per row: the key subsets' weights exp2(m_k - M) / L once, and the lse
  float* comb_w = comb_l + 4 * 16;  // [rows][KS]
  for (int r = tid; r < R; r += 128) {
    const int rgr = r >> 4, rr = r & 15;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < KS; ++k) M = fmaxf(M, comb_m[(rgr + k * RGN) * 16 + rr]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float wk[KS], L = 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      wk[k] = ex2f(comb_m[(rgr + k * RGN) * 16 + rr] - Mu);
      L += wk[k] * comb_l[(rgr + k * RGN) * 16 + rr];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k) comb_w[r * KS + k] = wk[k] * inv;
    const float lse = L > 0.f ? (Mu + __log2f(L)) * kLn2f : -INFINITY;
    if (!partial) {
      if (p.lse) p.lse[row_of(r)] = lse;
    } else {
      p.part_lse[it.part_row + r] = lse;
    }
  }
  asm volatile("bar.sync 2, 128;" ::: "memory");
  // O: four columns a thread at a time, a weighted sum over the key subsets
  constexpr int C4 = D / 4;
  for (int idx = tid; idx < R * C4; idx += 128) {
    const int r = idx / C4, c = idx % C4;
    const int rgr = r >> 4, rr = r & 15;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const float w = comb_w[r * KS + k];
      const float4 v = *reinterpret_cast<const float4*>(&comb_o[((rgr + k * RGN) * 16 + rr) * D + 4 * c]);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (!partial) {
      uint2 pk;
      pk.x = Elt<T>::from_f2(acc.x, acc.y);
      pk.y = Elt<T>::from_f2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(static_cast<T*>(p.out) + row_of(r) * D + 4 * c) = pk;
    } else {
      *reinterpret_cast<float4*>(p.part_o + (int64_t(it.part_row) + r) * D + 4 * c) = acc;
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
  pdl_wait();  // the partial states come from the attention kernels before it
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

// Stages of a decode launch: a launch of at most one CTA per SM streams each
// item through 192 KB of stages (one CTA per SM); larger launches keep two
// CTAs of kDecStages stages on an SM.  The bytes in flight per SM set the
// pace: the decode timing script's 128 items ran 15.8 us with one CTA of 3
// stages on each of 128 SMs and 14.6 us with 6, while batches of several
// waves ran 40 % slower with one CTA of 4 stages per SM than with two of 3.
template <int D>
constexpr int kDeepStages = (192 * 1024) / DecCfg<D>::STAGE;

template <typename T, int D, int G, int NST>
cudaError_t launch_cuda_cores_n(const RunArgs& a, const CUtensorMap* map, const KParams& kp, int use_tma) {
  using C = DecCfg<D, NST>;
  static std::atomic<uint64_t> attr_set{0};
  cudaError_t e = set_smem_once(attr_set, reinterpret_cast<const void*>(decode_kernel<T, D, G, NST>), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<T, D, G, NST>, unsigned(a.hp->n_dec), unsigned(kDecThreads), size_t(C::SMEM),
                    a.stream, *map, kp, use_tma);
}

template <typename T, int D, int G>
cudaError_t launch_cuda_cores(const RunArgs& a, const CUtensorMap* map, const KParams& kp, int use_tma) {
  if (a.hp->n_dec <= a.hp->num_sms) return launch_cuda_cores_n<T, D, G, kDeepStages<D>>(a, map, kp, use_tma);
  return launch_cuda_cores_n<T, D, G, kDecStages>(a, map, kp, use_tma);
}

template <typename T, int D, int RC, int NST>
cudaError_t launch_mma_n(const RunArgs& a, const CUtensorMap* map, const KParams& kp, int use_tma, int item0,
                         int n) {
  using C = DecCfg<D, NST>;
  static std::atomic<uint64_t> attr_set{0};
  cudaError_t e = set_smem_once(attr_set, reinterpret_cast<const void*>(decode_mma_kernel<T, D, RC, NST>), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_mma_kernel<T, D, RC, NST>, unsigned(n), unsigned(dm_threads<D, NST>()), size_t(C::SMEM), a.stream,
                    *map, kp, use_tma, item0);
}

template <typename T, int D, int RC>
cudaError_t launch_mma(const RunArgs& a, const CUtensorMap* map, const KParams& kp, int use_tma, int item0,
                       int n) {
  if (n <= a.hp->num_sms) return launch_mma_n<T, D, RC, kDeepStages<D>>(a, map, kp, use_tma, item0, n);
  return launch_mma_n<T, D, RC, kDecStages>(a, map, kp, use_tma, item0, n);
}

// The plan fixes the kernel: CUDA cores (one launch, every item a single
// query token at G <= 8), or the warp-MMA kernel with one launch per row
// class over that class's consecutive items.
template <typename T, int D>
cudaError_t launch_decode_d(const RunArgs& a, const CUtensorMap* map, const KParams& kp) {
  const HostPlan& hp = *a.hp;
  const int use_tma = (map != nullptr && hp.ps >= 8 && !a.force_cp_async) ? 1 : 0;
  CUtensorMap dummy;
  memset(&dummy, 0, sizeof(dummy));
  const CUtensorMap* m = use_tma ? map : &dummy;
  if (hp.dec_cores) {
    switch (hp.G) {
      case 1: return launch_cuda_cores<T, D, 1>(a, m, kp, use_tma);
      case 2: return launch_cuda_cores<T, D, 2>(a, m, kp, use_tma);
      case 4: return launch_cuda_cores<T, D, 4>(a, m, kp, use_tma);
      case 8: return launch_cuda_cores<T, D, 8>(a, m, kp, use_tma);
      default: return cudaErrorInvalidValue;
    }
  }
  if constexpr (D == 256) {
    return cudaErrorInvalidValue;  // no warp-MMA kernel at head_dim 256
  } else {
    int item0 = 0;
    for (int c = 0; c < kDecClasses; ++c) {
      const int n = hp.n_dec_class[c];
      if (n == 0) continue;
      cudaError_t e = cudaSuccess;
      switch (c) {
        case 0: e = launch_mma<T, D, 0>(a, m, kp, use_tma, item0, n); break;
        case 1: e = launch_mma<T, D, 1>(a, m, kp, use_tma, item0, n); break;
        case 2: e = launch_mma<T, D, 2>(a, m, kp, use_tma, item0, n); break;
        default: e = cudaErrorInvalidValue; break;  // 64-row items go to the prefill kernel
      }
      if (e != cudaSuccess) return e;
      item0 += n;
    }
    return item0 == hp.n_dec ? cudaSuccess : cudaErrorInvalidValue;
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
    return bf ? launch_decode_d<__nv_bfloat16, 128>(a, map_rows, kp)
              : launch_decode_d<__half, 128>(a, map_rows, kp);
  if (a.hp->D == 256)
    return bf ? launch_decode_d<__nv_bfloat16, 256>(a, map_rows, kp)
              : launch_decode_d<__half, 256>(a, map_rows, kp);
  return bf ? launch_decode_d<__nv_bfloat16, 64>(a, map_rows, kp)
            : launch_decode_d<__half, 64>(a, map_rows, kp);
}

cudaError_t launch_merge(const RunArgs& a) {
  if (a.hp->n_merge == 0) return cudaSuccess;
  KParams kp = make_params(a);
  const int rows = a.hp->n_merge * a.hp->G;
  const int blocks = (rows + 7) / 8;
  const bool bf = a.hp->dtype == PA_BF16;
  const unsigned nb = unsigned(blocks);
  if (a.hp->D == 128)
    return bf ? launch_pdl(merge_kernel<__nv_bfloat16, 128>, nb, 256u, size_t(0), a.stream, kp, rows)
              : launch_pdl(merge_kernel<__half, 128>, nb, 256u, size_t(0), a.stream, kp, rows);
  if (a.hp->D == 256)
    return bf ? launch_pdl(merge_kernel<__nv_bfloat16, 256>, nb, 256u, size_t(0), a.stream, kp, rows)
              : launch_pdl(merge_kernel<__half, 256>, nb, 256u, size_t(0), a.stream, kp, rows);
  return bf ? launch_pdl(merge_kernel<__nv_bfloat16, 64>, nb, 256u, size_t(0), a.stream, kp, rows)
            : launch_pdl(merge_kernel<__half, 64>, nb, 256u, size_t(0), a.stream, kp, rows);
}

cudaError_t launch_debug_gather(const RunArgs& a, int32_t* page_out, int32_t* slot_out) {
  if (a.hp->B == 0) return cudaSuccess;
  KParams kp = make_params(a);
  debug_gather_kernel<<<a.hp->B, 256, 0, a.stream>>>(kp, a.hp->B, page_out, slot_out);
  return cudaGetLastError();
}

}  // namespace pa
