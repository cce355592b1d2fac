// Tensor-core prefill kernel over the paged KV cache (sm_103a: tcgen05 + TMEM).
//
// One CTA handles one work item: 128 packed query rows (128/G consecutive
// tokens x the G query heads of one kv head, head-minor) of one request,
// against the key range [kv_tok0, kv_tok1) of that request.  Packing the G
// heads of a group into the MMA's M dimension makes every K/V tile load serve
// all G heads (grouped-query attention has the higher operational intensity
// the FlashInfer issue "How are prefill and decode kernels different?"
// points out).  Key tiles wholly past the causal diagonal of the tile's last
// row are never visited: the planner stops the range there ("skips the fully
// masked out tails", llama.cpp discussion "Pad for prefill stage?").
//
// Warp roles (192 threads):
//   warps 0-3  softmax / correction / epilogue; thread i owns row i, which is
//              TMEM lane i, so the online softmax needs no shuffles.
//   warp 4     producer: gathers the tile's pages through the page table with
//              TMA (4-D tensor map over the cache, 128-byte swizzle), or with
//              cp.async for pages smaller than 8 slots.
//   warp 5     MMA issuer (one thread) and TMEM owner.
//
// TMEM (512 columns): S double buffer at columns 0 and 128 (fp32 128x128),
// O at column 256 (fp32 128xD).  P goes through shared memory as the A
// operand of the second MMA.
//
// Per key tile j:  S_j = Q K_j^T (tcgen05, both K-major) -> softmax threads
// load S_j, mask the diagonal / tail, update the running max m and sum l,
// write P_j (fp16/bf16) -> O += P_j V_j (V as an MN-major B operand).  The
// running max is only moved (and O rescaled in TMEM) when it grows by more
// than 8 in log2 units; p stays below 2^8 in between, which fp32 sums and
// fp16/bf16 P carry without loss of range.  S_{j+1} is issued before PV_j so
// the tensor core works while the softmax threads run.
//
// Rows that see only a handful of keys average nothing out, so the 8-bit
// mantissa of a bf16 P would show in their output.  All such rows sit in the
// first key tile of a sequence; there P is written as hi + lo (two fp16/bf16
// halves, lo = p - hi) and PV is issued for both, which gives P about 16
// mantissa bits where it matters for one extra MMA set per item.
#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr int kPreThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kColS0 = 0, kColO = 256;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct PreCfg {
  static constexpr int NKB = D / 64;                 // 128-byte column blocks of a row
  static constexpr int NST = (D == 128) ? 2 : 4;     // K/V pipeline stages
  static constexpr int BLK = 128 * 128;              // one 128-row x 128-byte block
  static constexpr int Q_BYTES = NKB * BLK;
  static constexpr int KV_BYTES = NKB * BLK;         // 128 keys of K (or V)
  static constexpr int P_BYTES = 2 * BLK;            // 128 rows x 128 keys x 2 bytes
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NST * KV_BYTES;
  static constexpr int OFF_PLO = OFF_P + P_BYTES;    // low half of split P (first key tile)
  static constexpr int OFF_BAR = OFF_PLO + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // barriers + alignment slack
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait, made uniform across the warp (all lanes leave together).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status) {
  bool ok = mbar_wait(bar, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Wait that ignores the abort flag (used to drain in-flight async work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > PA_WAIT_LIMIT_CYCLES) break;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kPreThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const KParams p, const int use_tma) {
  using C = PreCfg<D>;
  constexpr int NKB = C::NKB, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_addr = sbase + C::OFF_Q;
  const uint32_t p_addr = sbase + C::OFF_P;
  const uint32_t plo_addr = sbase + C::OFF_PLO;
  auto k_addr = [&](int st) { return sbase + C::OFF_K + st * C::KV_BYTES; };
  auto v_addr = [&](int st) { return sbase + C::OFF_V + st * C::KV_BYTES; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* full = bars;              // [NST] K/V tile landed
  uint64_t* empty = bars + NST;       // [NST] PV MMA done with the stage
  uint64_t* s_full = bars + 2 * NST;  // [2] S MMA done
  uint64_t* s_free = s_full + 2;      // [2] softmax warps have read S
  uint64_t* p_full = s_free + 2;      // P (and O correction) written
  uint64_t* o_done = p_full + 1;      // PV MMA done
  uint64_t* q_full = o_done + 1;      // Q staged
  uint64_t* fin = q_full + 1;         // all MMAs retired (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 16);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PreItem it = p.pre[blockIdx.x];
  const ReqEntry rq = p.req[it.req];
  const int nkt = (it.kv_tok1 - it.kv_tok0 + kKvTile - 1) / kKvTile;
  // split P on the first key tile when some row of the item sees < 128 keys
  const int first_vis = p.causal ? (rq.kv_len - rq.qo_len + it.q_tok0 + 1) : rq.kv_len;
  const bool lo_split0 = (it.kv_tok0 == 0) && (first_vis < kKvTile);

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full[i], use_tma ? 1 : 32);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(q_full, 4);
    mbar_init(fin, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 5) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (use_tma && lane == 0) tma_prefetch_desc(&kv_map);
    const int ps = p.ps, sh = p.ps_shift;
    int issued = 0;
    for (int j = 0; j < nkt; ++j) {
      const int st = j % NST;
      if (j >= NST) {
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[st], ((j / NST) - 1) & 1, abort_flag, p.status);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
      const int k0 = it.kv_tok0 + j * kKvTile;
      const int kend = min(k0 + kKvTile, it.kv_tok1);
      if (use_tma) {
        const int pg0 = k0 >> sh;
        const int npg = ((kend - 1) >> sh) - pg0 + 1;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(npg * ps * 128 * NKB * 2));
        __syncwarp();
        for (int l = lane; l < npg; l += 32) {
          const KvLoc loc = kv_locate(p.pages, rq.page_start, k0 + l * ps, sh);
          int pid = loc.page;
          if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
            atomicOr(p.status, PA_DEV_BAD_INDEX);
            pid = 0;
          }
#pragma unroll
          for (int kb = 0; kb < NKB; ++kb) {
            tma_load_4d(k_addr(st) + kb * C::BLK + l * ps * 128, &kv_map, kb * 64, it.kv_head, 0, 2 * pid,
                        &full[st]);
            tma_load_4d(v_addr(st) + kb * C::BLK + l * ps * 128, &kv_map, kb * 64, it.kv_head, 0, 2 * pid + 1,
                        &full[st]);
          }
        }
      } else {
        const T* kvb = static_cast<const T*>(p.kv);
        for (int t = lane; t < kKvTile; t += 32) {
          const int tok = k0 + t;
          const bool valid = tok < kend;
          const T* srck = kvb;
          const T* srcv = kvb;
          if (valid) {
            const KvLoc loc = kv_locate(p.pages, rq.page_start, tok, sh);
            int pid = loc.page;
            if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
              atomicOr(p.status, PA_DEV_BAD_INDEX);
              pid = 0;
            }
            const size_t rowk = ((size_t(pid) * 2 * ps + loc.slot) * p.Hkv + it.kv_head) * D;
            srck = kvb + rowk;
            srcv = kvb + rowk + size_t(ps) * p.Hkv * D;
          }
#pragma unroll
          for (int kb = 0; kb < NKB; ++kb) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t off = kb * C::BLK + t * 128 + ((c ^ (t & 7)) * 16);
              cp_async16(k_addr(st) + off, srck + (valid ? kb * 64 + c * 8 : 0), valid ? 16u : 0u);
              cp_async16(v_addr(st) + off, srcv + (valid ? kb * 64 + c * 8 : 0), valid ? 16u : 0u);
            }
          }
        }
        cp_async_commit();
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(&full[st]);
      }
      issued = j + 1;
    }
    // drain: copies still in flight must land before the CTA's memory goes away
    if (use_tma && lane == 0) {
      for (int j = max(0, issued - NST); j < issued; ++j) drain_wait(&full[j % NST], (j / NST) & 1);
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(Elt<T>::kBf16, 0, 0, 128, 128);
      const uint32_t id_o = idesc_f16(Elt<T>::kBf16, 0, 1, 128, D);
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
      tc_fence_after();
      for (int j = 0; ok && j <= nkt; ++j) {
        if (j < nkt) {
          const int st = j % NST;
          ok = mbar_wait(&full[st], (j / NST) & 1, abort_flag, p.status);
          if (ok && j >= 2) ok = mbar_wait(&s_free[j & 1], ((j >> 1) - 1) & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + kColS0 + (j & 1) * 128;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t koff = (k >> 2) * C::BLK + (k & 3) * 32;
            tc_mma_ss(d, smem_desc_sw128(q_addr + koff, 16, 1024), smem_desc_sw128(k_addr(st) + koff, 16, 1024),
                      id_s, k > 0 ? 1u : 0u);
          }
          tc_commit(&s_full[j & 1]);
        }
        if (j >= 1) {
          const int i = j - 1, st = i % NST;
          ok = mbar_wait(p_full, i & 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kKvTile / 16; ++k) {
            const uint32_t aoff = (k >> 2) * C::BLK + (k & 3) * 32;
            tc_mma_ss(tmem + kColO, smem_desc_sw128(p_addr + aoff, 16, 1024),
                      smem_desc_sw128(v_addr(st) + k * 2048, C::BLK, 1024), id_o, (i > 0 || k > 0) ? 1u : 0u);
          }
          if (i == 0 && lo_split0) {
#pragma unroll
            for (int k = 0; k < kKvTile / 16; ++k) {
              const uint32_t aoff = (k >> 2) * C::BLK + (k & 3) * 32;
              tc_mma_ss(tmem + kColO, smem_desc_sw128(plo_addr + aoff, 16, 1024),
                        smem_desc_sw128(v_addr(st) + k * 2048, C::BLK, 1024), id_o, 1u);
            }
          }
          tc_commit(&empty[st]);
          tc_commit(o_done);
        }
      }
      tc_commit(fin);
      drain_wait(fin, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int r = tid;
    const int G = p.G;
    const int tok_local = r >> p.g_shift;
    const int g = r & (G - 1);
    const bool row_valid = tok_local < it.q_ntok;
    const int qi = it.q_tok0 + tok_local;
    const int64_t qrow = (int64_t(rq.qo_start) + qi) * p.Hq + int64_t(it.kv_head) * G + g;

    {  // stage this row of Q (zeros for rows past the tile)
      const T* qsrc = static_cast<const T*>(p.q) + (row_valid ? qrow * D : 0);
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
        for (int c = 0; c < 8; ++c)
          cp_async16(q_addr + kb * C::BLK + r * 128 + ((c ^ (r & 7)) * 16), qsrc + (row_valid ? kb * 64 + c * 8 : 0),
                     row_valid ? 16u : 0u);
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);
    }

    int row_end = p.causal ? (rq.kv_len - rq.qo_len + qi + 1) : rq.kv_len;
    row_end = min(row_end, it.kv_tok1);
    if (!row_valid) row_end = 0;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l_sum = 0.f;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;

    for (int j = 0; j < nkt; ++j) {
      const int k0 = it.kv_tok0 + j * kKvTile;
      ok = warp_wait(&s_full[j & 1], (j >> 1) & 1, abort_flag, p.status);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      const uint32_t sa = tmem + lane_base + kColS0 + (j & 1) * 128;
      tmem_ld32(sa + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
      tmem_ld32(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
      tmem_ld32(sa + 64, *reinterpret_cast<uint32_t(*)[32]>(s + 64));
      tmem_ld32(sa + 96, *reinterpret_cast<uint32_t(*)[32]>(s + 96));
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 128; ++i) asm volatile("" : "+r"(s[i]));
      const bool lo_split = lo_split0 && j == 0;
      if (!lo_split) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[j & 1]);
      }

      // mask (diagonal / tail tiles only) and tile max
      const int lim = row_end - k0;
      float mx = -INFINITY;
      if (lim >= kKvTile) {
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float v = (c < lim) ? __uint_as_float(s[c]) : -INFINITY;
          s[c] = __float_as_uint(v);
          mx = fmaxf(mx, v);
        }
      }
      const float mx2 = mx * sl2;
      float alpha = 1.f;
      bool resc = false;
      if (mx2 > m_ref + 8.f) {
        if (m_ref != -INFINITY) {
          alpha = ex2(m_ref - mx2);
          resc = true;
        }
        m_ref = mx2;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs = 0.f;
      uint32_t pw[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float a = ex2(fmaf(__uint_as_float(s[2 * c]), sl2, -m_use));
        const float b = ex2(fmaf(__uint_as_float(s[2 * c + 1]), sl2, -m_use));
        rs += a + b;
        pw[c] = Elt<T>::from_f2(a, b);
      }
      l_sum = l_sum * alpha + rs;

      // PV of the previous tile must be done before P and O are touched
      if (j >= 1) {
        ok = warp_wait(o_done, (j - 1) & 1, abort_flag, p.status);
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + kColO + c4 * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_base + kColO + c4 * 32, o);
        }
        tmem_wait_st();
      }
      // keys past the end of the range: zero their V rows (they may hold
      // anything, and 0 * NaN would poison O); cp.async already zero-filled
      if (use_tma && j == nkt - 1) {
        const int valid = it.kv_tok1 - k0;
        if (valid < kKvTile) {
          const int st = j % NST;
          ok = warp_wait(&full[st], (j / NST) & 1, abort_flag, p.status);
          if (!ok) break;
          if (r >= valid) {
            uint8_t* vrow = smem + C::OFF_V + st * C::KV_BYTES + r * 128;
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vrow + kb * C::BLK + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // P row -> shared memory, K-major with the 128-byte swizzle
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v = make_uint4(pw[kb * 32 + c * 4 + 0], pw[kb * 32 + c * 4 + 1], pw[kb * 32 + c * 4 + 2],
                               pw[kb * 32 + c * 4 + 3]);
          *reinterpret_cast<uint4*>(smem + C::OFF_P + kb * C::BLK + r * 128 + ((c ^ (r & 7)) * 16)) = v;
        }
      if (lo_split) {
        // second pass over S (still in TMEM: its buffer is only released
        // below): the same p values again, minus their rounded high halves
        tmem_ld32(sa + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
        tmem_ld32(sa + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
        tmem_ld32(sa + 64, *reinterpret_cast<uint32_t(*)[32]>(s + 64));
        tmem_ld32(sa + 96, *reinterpret_cast<uint32_t(*)[32]>(s + 96));
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) asm volatile("" : "+r"(s[i]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[j & 1]);
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t lw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int col = kb * 64 + c * 8 + 2 * u;
              const float va = (col < lim) ? __uint_as_float(s[col]) : -INFINITY;
              const float vb = (col + 1 < lim) ? __uint_as_float(s[col + 1]) : -INFINITY;
              const float a = ex2(fmaf(va, sl2, -m_use));
              const float b = ex2(fmaf(vb, sl2, -m_use));
              const float2 hi = Elt<T>::to_f2(Elt<T>::from_f2(a, b));
              lw[u] = Elt<T>::from_f2(a - hi.x, b - hi.y);
            }
            *reinterpret_cast<uint4*>(smem + C::OFF_PLO + kb * C::BLK + r * 128 + ((c ^ (r & 7)) * 16)) =
                make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }

    // ---------------------------------------------------------------- epilogue
    if (ok) ok = warp_wait(o_done, (nkt - 1) & 1, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const float lse_v = l_sum > 0.f ? (m_use + __log2f(l_sum)) * kLn2 : -INFINITY;
      const bool partial = it.part_row >= 0;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kColO + c4 * 32, o);
        tmem_wait_ld(o);
        if (row_valid) {
          if (!partial) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + qrow * D + c4 * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = Elt<T>::from_f2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
              w.y = Elt<T>::from_f2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
              w.z = Elt<T>::from_f2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
              w.w = Elt<T>::from_f2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
              dst[v] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + (int64_t(it.part_row) + r) * D + c4 * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                   __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
          }
        }
      }
      if (row_valid) {
        if (!partial) {
          if (p.lse) p.lse[qrow] = lse_v;
        } else {
          p.part_lse[it.part_row + r] = lse_v;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <typename T, int D>
cudaError_t launch_prefill_t(const RunArgs& a, const CUtensorMap* map, const KParams& kp, int use_tma) {
  using C = PreCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  prefill_kernel<T, D><<<a.hp->n_pre, kPreThreads, C::SMEM, a.stream>>>(*map, kp, use_tma);
  return cudaGetLastError();
}

}  // namespace

KParams make_params(const RunArgs& a);

cudaError_t launch_prefill(const RunArgs& a, const CUtensorMap* map_sw128) {
  if (a.hp->n_pre == 0) return cudaSuccess;
  KParams kp = make_params(a);
  kp.n_items = a.hp->n_pre;
  const int use_tma = (map_sw128 != nullptr && !a.force_cp_async && a.hp->ps >= 8) ? 1 : 0;
  CUtensorMap dummy;
  const CUtensorMap* m = use_tma ? map_sw128 : &dummy;
  if (!use_tma) memset(&dummy, 0, sizeof(dummy));
  const bool bf = a.hp->dtype == PA_BF16;
  if (a.hp->D == 128)
    return bf ? launch_prefill_t<__nv_bfloat16, 128>(a, m, kp, use_tma) : launch_prefill_t<__half, 128>(a, m, kp, use_tma);
  return bf ? launch_prefill_t<__nv_bfloat16, 64>(a, m, kp, use_tma) : launch_prefill_t<__half, 64>(a, m, kp, use_tma);
}

}  // namespace pa
