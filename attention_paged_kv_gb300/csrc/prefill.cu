// Tensor-core prefill kernel over the paged KV cache (sm_103a: tcgen05 + TMEM).
//
// One CTA handles one work item: 256 packed query rows -- 256/G consecutive
// tokens x the G query heads of one kv head, head-minor -- of one request,
// against the key range [kv_tok0, kv_tok1) of that request.  The rows form
// two 128-row MMA tiles, A and B, that share every K/V tile load, as do the G
// heads of a group (grouped-query attention has the higher operational
// intensity the FlashInfer issue "How are prefill and decode kernels
// different?" points out).  Key tiles wholly past the causal diagonal of the
// item's last row are never visited: the planner stops the range there
// ("skips the fully masked out tails", llama.cpp discussion "Pad for prefill
// stage?").
//
// Warp roles (352 threads):
//   warps 0-3  softmax / correction / epilogue of tile A; thread i owns row i
//              = TMEM lane i, so the online softmax needs no shuffles.
//   warps 4-7  the same for tile B.
//   warp 8     K producer: TMA loads of the two Q tiles (3-D map over q) and
//              of each key tile's K pages through the page table (4-D map
//              over the cache, 128-byte swizzle), or cp.async for pages of
//              < 8 slots.
//   warp 9     MMA issuer (one thread) and TMEM owner.
//   warp 10    V producer: the same for each key tile's V pages.
//
// K and V tiles have separate two-slot rings (four for head_dim 64), so the
// next K tile loads as soon as both S MMAs have read the slot it reuses.  The
// producer reads each tile's page ids two tiles ahead: with the page-table
// read between a slot becoming free and its copy, the producer had set the
// pace of the whole CTA (a key-tile period of ~4000 SM cycles against ~3700).
//
// TMEM (512 columns): S_A at 0, S_B at 128 (fp32 128x128), O_A at 256, O_B at
// 384 (fp32 128xD).  P (fp16/bf16, two per column) is written over the first
// 64 columns of its S and feeds the PV MMA as a TMEM A operand.
//
// The one-tile variant (template NT = 1: 128-row items, 192 threads, S at
// TMEM column 0 and O at 128, one K/V stage) serves head_dim 256, whose O
// takes 256 columns a tile, and batches of short prompts, where two CTAs to
// an SM hide each other's fixed costs (Q and first K/V loads, epilogue).
//
// Per key tile j the MMA thread (which polls its barriers rather than
// sleeping on them) issues, in order:
//   PV_A(j) ; S_A(j+1) ; PV_B(j) ; S_B(j+1)
// so while the softmax warps of one tile turn S into P, the tensor core works
// on the other tile.  Softmax per tile: the S row is read from TMEM into
// registers (four loads, one wait), then max, exp2, the row sum and P.
// The running max is only moved (and O rescaled in TMEM) when it grows by
// more than 8 in log2 units; p stays below 2^8 in between, which fp32 sums
// and fp16/bf16 P carry without loss of range.
//
// Rows that see only a handful of keys average nothing out, so the 8-bit
// mantissa of a bf16 P would show in their output.  All such rows sit in the
// first key tile of a sequence; there P is split into hi (TMEM) + lo = p - hi
// (shared memory) and PV is issued for both, which gives P about 16 mantissa
// bits where it matters.
#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace pa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

// NT = 128-row Q tiles per CTA.  Two tiles (the default) share every K/V
// load and take turns on the tensor core; one tile at D = 256, where O alone
// takes 256 TMEM columns a tile, and for batches of short prompts, where one
// tile per CTA lets two CTAs share an SM and hide each other's fixed costs.
template <int D, int NT>
struct PreCfg {
  static_assert(NT == 1 || (NT == 2 && D <= 128), "two tiles need 2 x (128 + D) <= 512 TMEM columns");
  // producers: two tiles have one warp for K and one for V (each TMA copy
  // costs its issuing thread ~90 cycles, and one warp issuing all of a key
  // tile's copies set the pace); one tile keeps one producer warp, so that
  // two CTAs of 6 warps still fit an SM at 168 registers a thread
  static constexpr int PRODS = NT == 2 ? 2 : 1;
  static constexpr int THREADS = 32 * (4 * NT + 1 + PRODS);  // softmax warpgroup(s), MMA issuer, producer(s)
  static constexpr int WARP_PROD = 4 * NT, WARP_MMA = 4 * NT + 1;
  static constexpr int WARP_PROD_V = PRODS == 2 ? 4 * NT + 2 : WARP_PROD;
  static constexpr int NKB = D / 64;                 // 128-byte column blocks of a row
  static constexpr int NST = NT == 1 ? 1 : (D == 128 ? 2 : 4);  // K/V pipeline stages
  static constexpr int BLK = 128 * 128;              // one 128-row x 128-byte block
  static constexpr int Q_BYTES = NKB * BLK;          // one 128-row Q tile
  static constexpr int KV_BYTES = NKB * BLK;         // 128 keys of K (or V)
  static constexpr int P_BYTES = 2 * BLK;            // 128 rows x 128 keys x 2 bytes
  static constexpr int OFF_Q = 0;                    // tiles A, B
  static constexpr int OFF_K = NT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NST * KV_BYTES;
  static constexpr int OFF_FREE = OFF_V + NST * KV_BYTES;
  // P_lo buffers for the first key tile: tile A reuses K stage 0 when it is
  // large enough (its keys are consumed by both S MMAs before P is written)
  static constexpr int OFF_PLO_A = (KV_BYTES >= P_BYTES) ? OFF_K : OFF_FREE;
  static constexpr int OFF_PLO_B = (KV_BYTES >= P_BYTES) ? OFF_FREE : OFF_FREE + P_BYTES;
  static constexpr int OFF_BAR = (NT == 1) ? (OFF_PLO_A == OFF_FREE ? OFF_FREE + P_BYTES : OFF_FREE)
                                           : OFF_PLO_B + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // barriers + alignment slack
  // TMEM: S_x at columns 128 x, O_x after the S columns
  static constexpr int O_COL = NT * 128;
  static constexpr uint32_t TMEM_COLS = (NT * (128 + D) <= 256) ? 256u : 512u;
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(NT == 2 || D == 256 || 2 * (SMEM + 1024) <= 233472, "two one-tile CTAs share an SM");
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bounded wait, made uniform across the warp (all lanes leave together).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status, long long limit) {
  bool ok = mbar_wait(bar, parity, abort_flag, status, limit);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that polls with non-blocking probes and never suspends: the
// MMA thread waits this way, since waking a suspended thread cost ~1.8 % of
// the prefill (the softmax warps, which share their SM sub-partitions with the
// other tile's softmax, wait with try_wait: spinning there cost 3.6 %, and
// neither a suspend-time hint for them nor a back-off for the MMA thread
// changed anything).
__device__ __forceinline__ bool spin_wait(uint64_t* bar, uint32_t parity, volatile int32_t* abort_flag,
                                          int32_t* status, long long limit) {
  const uint32_t a = smem_u32(bar);
  if (mbar_test_wait(a, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_test_wait(a, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      *abort_flag = 1;
      atomicOr(status, PA_DEV_TIMEOUT);
      return false;
    }
  }
}
// Wait that ignores the abort flag (used to drain in-flight async work).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const long long t0 = clock64();
  while (!mbar_try_wait(a, parity)) {
    if (clock64() - t0 > PA_WAIT_LIMIT_CYCLES) break;
  }
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <typename T, int D, int NT>
__global__ void __launch_bounds__(PreCfg<D, NT>::THREADS, NT == 1 ? 2 : 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap o_map, const __grid_constant__ CUtensorMap o32_map,
                   const KParams p, const int use_tma) {
  using C = PreCfg<D, NT>;
  constexpr int NKB = C::NKB, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto q_addr = [&](int x) { return sbase + C::OFF_Q + x * C::Q_BYTES; };
  auto k_addr = [&](int st) { return sbase + C::OFF_K + st * C::KV_BYTES; };
  auto v_addr = [&](int st) { return sbase + C::OFF_V + st * C::KV_BYTES; };
  auto plo_off = [&](int x) { return x == 0 ? C::OFF_PLO_A : C::OFF_PLO_B; };

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  // K and V have their own stages: a K slot is free once both S MMAs have
  // read it, long before the PV MMAs are done with the V of the same tile
  uint64_t* full_k = bars;              // [NST] K tile landed
  uint64_t* full_v = bars + NST;        // [NST] V tile landed
  uint64_t* empty_k = bars + 2 * NST;   // [NST] both S MMAs done with the K slot
  uint64_t* empty_v = bars + 3 * NST;   // [NST] both PV MMAs done with the V slot
  uint64_t* q_full = bars + 4 * NST;    // both Q tiles landed
  uint64_t* s_full = q_full + 1;        // [2] S_x MMA done
  uint64_t* p_full = s_full + 2;        // [2] P_x (and O_x correction) written
  uint64_t* o_done = p_full + 2;        // [2] the last PV_x MMA done (one phase)
  uint64_t* fin = o_done + 2;           // all MMAs retired (teardown)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  uint64_t* never = bars + 25;          // test hook: a barrier nothing completes
  uint64_t* o_st = bars + 26;           // [2] tile x's O staged in shared memory (its 4 warps)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PreItem it = p.pre[blockIdx.x];
  const ReqEntry rq = p.req[it.req];
  const int G = p.G;
  const int TQ = kQRows >> p.g_shift;           // tokens per 128-row tile
  const bool has_b = NT == 2 && it.q_ntok > TQ;
  const int nkt = (it.kv_tok1 - it.kv_tok0 + kKvTile - 1) / kKvTile;
  // split P on the first key tile when some row of the item sees < 128 keys
  const int first_vis = p.causal ? (rq.kv_len - rq.qo_len + it.q_tok0 + 1) : rq.kv_len;
  const bool lo_split0 = (it.kv_tok0 == 0) && (first_vis < kKvTile);

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_k[i], use_tma ? 1 : 32);
      mbar_init(&full_v[i], use_tma ? 1 : 32);
      mbar_init(&empty_k[i], 1);
      mbar_init(&empty_v[i], 1);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(fin, 1);
    mbar_init(never, 1);
    mbar_init(&o_st[0], 4);
    mbar_init(&o_st[1], 4);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == C::WARP_MMA) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::WARP_PROD || warp == C::WARP_PROD_V) {
    // ---------------------------------------------------------------- producer(s)
    // halves [h0, h1) of each key tile: 0 = K, 1 = V
    const int h0 = (C::PRODS == 2 && warp == C::WARP_PROD_V) ? 1 : 0;
    const int h1 = (C::PRODS == 2 && warp == C::WARP_PROD) ? 1 : 2;
    if (warp == C::WARP_PROD && lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&o_map);
      tma_prefetch_desc(&o32_map);
      if (use_tma) tma_prefetch_desc(&kv_map);
    }
    const int ps = p.ps, sh = p.ps_shift;
    // TMA path: lane l gathers page l of every key tile (at most 16 pages of
    // >= 8 slots).  Its page id is read two tiles ahead, so that no global
    // load sits between a slot becoming free and the copy into it: with the
    // load in between, the producer set the pace of the whole CTA.
    auto tile_pid = [&](int jj) -> int {
      if (!use_tma || jj >= nkt) return 0;
      const int k0j = it.kv_tok0 + jj * kKvTile;
      const int kendj = min(k0j + kKvTile, it.kv_tok1);
      const int npgj = ((kendj - 1) >> sh) - (k0j >> sh) + 1;
      return lane < npgj ? __ldg(p.pages + rq.page_start + (k0j >> sh) + lane) : 0;
    };
    int pid_j = tile_pid(0), pid_j1 = tile_pid(1);
    pdl_wait();  // q and the cache may come from the previous kernel on the stream
    if (warp == C::WARP_PROD && lane == 0) {
      mbar_arrive_expect_tx(q_full, uint32_t((has_b ? 2 : 1) * C::Q_BYTES));
#pragma unroll
      for (int kb = 0; kb < NKB; ++kb) {
        tma_load_3d(q_addr(0) + kb * C::BLK, &q_map, kb * 64, it.kv_head * G, rq.qo_start + it.q_tok0, q_full);
        if (has_b)
          tma_load_3d(q_addr(1) + kb * C::BLK, &q_map, kb * 64, it.kv_head * G, rq.qo_start + it.q_tok0 + TQ,
                      q_full);
      }
    }
    int issued_k = 0, issued_v = 0;
    bool ok = true;
    for (int j = 0; ok && j < nkt; ++j) {
     {
      const int st = j % NST;
      const int k0 = it.kv_tok0 + j * kKvTile;
      const int kend = min(k0 + kKvTile, it.kv_tok1);
      const int pid_j2 = tile_pid(j + 2);
      int pid = pid_j;
      if (use_tma && static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
        atomicOr(p.status, PA_DEV_BAD_INDEX);
        pid = 0;
      }
      pid_j = pid_j1;
      pid_j1 = pid_j2;
      for (int half = h0; half < h1 && ok; ++half) {  // 0: K, 1: V
        uint64_t* empty = half ? empty_v : empty_k;
        uint64_t* full = half ? full_v : full_k;
        const uint32_t dst0 = half ? v_addr(st) : k_addr(st);
        if (j >= NST) {
          if (lane == 0) ok = mbar_wait(&empty[st], ((j / NST) - 1) & 1, abort_flag, p.status, p.wait_limit);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        if (use_tma) {
          const int pg0 = k0 >> sh;
          const int npg = ((kend - 1) >> sh) - pg0 + 1;
          if (lane == 0) mbar_arrive_expect_tx(&full[st], uint32_t(npg * ps * 128 * NKB));
          __syncwarp();
          if (lane < npg) {
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb)
              tma_kv_rows(dst0 + kb * C::BLK + lane * ps * 128, &kv_map, kb * 64, it.kv_head, 0, 2 * pid + half,
                          &full[st], p.hnd);
          }
        } else {
          const T* kvb = static_cast<const T*>(p.kv);
          for (int t = lane; t < kKvTile; t += 32) {
            const int tok = k0 + t;
            const bool valid = tok < kend;
            const T* src = kvb;
            if (valid) {
              const KvLoc loc = kv_locate(p.pages, rq.page_start, tok, sh);
              int pid = loc.page;
              if (static_cast<unsigned>(pid) >= static_cast<unsigned>(p.num_pages)) {
                atomicOr(p.status, PA_DEV_BAD_INDEX);
                pid = 0;
              }
              src = kvb + kv_row(p, pid, half, loc.slot, it.kv_head) * D;
            }
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const uint32_t off = kb * C::BLK + t * 128 + ((c ^ (t & 7)) * 16);
                cp_async16(dst0 + off, src + (valid ? kb * 64 + c * 8 : 0), valid ? 16u : 0u);
              }
            }
          }
          cp_async_commit();
          cp_async_wait_all();
          fence_proxy_async_smem();
          mbar_arrive(&full[st]);
        }
        if (half) issued_v = j + 1; else issued_k = j + 1;
      }
     }
    }
    // drain: copies still in flight must land before the CTA's memory goes away
    if (lane == 0) {
      if (warp == C::WARP_PROD) drain_wait(q_full, 0);
      if (use_tma) {
        for (int j = max(0, issued_k - NST); j < issued_k; ++j) drain_wait(&full_k[j % NST], (j / NST) & 1);
        for (int j = max(0, issued_v - NST); j < issued_v; ++j) drain_wait(&full_v[j % NST], (j / NST) & 1);
      }
    }
    __syncwarp();
  } else if (warp == C::WARP_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(Elt<T>::kBf16, 0, 0, 128, 128);
      const uint32_t id_o = idesc_f16(Elt<T>::kBf16, 0, 1, 128, D);
      // Matrix descriptors of each operand's first k-step, made once: a
      // k-step (or another tile or stage) adds its byte offset / 16 to the
      // start-address field (shared addresses stay below 2^18, so the sum
      // never carries out of the field).
      const uint64_t dq0 = smem_desc_sw128(q_addr(0), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(k_addr(0), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(v_addr(0), C::BLK, 1024);
      auto issue_s = [&](int x, int st) {
        const uint32_t d = tmem + x * 128;
        const uint64_t qd = dq0 + uint64_t(x) * (C::Q_BYTES >> 4);
        const uint64_t kd = dk0 + uint64_t(st) * (C::KV_BYTES >> 4);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t koff = ((k >> 2) * C::BLK + (k & 3) * 32) >> 4;
          tc_mma_ss(d, qd + koff, kd + koff, id_s, k > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[x]);
      };
      auto issue_pv = [&](int x, int j, int st) {
        const uint32_t d = tmem + C::O_COL + x * 128;
        const uint64_t vd = dv0 + uint64_t(st) * (C::KV_BYTES >> 4);
#pragma unroll
        for (int k = 0; k < kKvTile / 16; ++k)
          tc_mma_ts(d, tmem + x * 128 + k * 8, vd + (k * 2048 >> 4), id_o, (j > 0 || k > 0) ? 1u : 0u);
        if (j == 0 && lo_split0) {
          const uint32_t lo = sbase + plo_off(x);
#pragma unroll
          for (int k = 0; k < kKvTile / 16; ++k) {
            const uint32_t aoff = (k >> 2) * C::BLK + (k & 3) * 32;
            tc_mma_ss(d, smem_desc_sw128(lo + aoff, 16, 1024), vd + (k * 2048 >> 4), id_o, 1u);
          }
        }
        if (j == nkt - 1) tc_commit(&o_done[x]);  // the epilogue's only wait on O
      };
      // tile A's P_lo of the first key tile may live in K slot 0: then that
      // slot is released only once PV_A(0) has read it
      const bool plo_in_k = lo_split0 && (C::OFF_PLO_A == C::OFF_K);
      bool ok = p.stall ? spin_wait(never, 0, abort_flag, p.status, p.wait_limit) : true;
      if (ok) ok = spin_wait(q_full, 0, abort_flag, p.status, p.wait_limit);
      if (ok) ok = spin_wait(&full_k[0], 0, abort_flag, p.status, p.wait_limit);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (has_b) issue_s(1, 0);
        if (!plo_in_k) tc_commit(&empty_k[0]);
      }
      for (int j = 0; ok && j < nkt; ++j) {
        const int st = j % NST;
        const bool more = j + 1 < nkt;
        const int st1 = (j + 1) % NST;
        ok = spin_wait(&p_full[0], j & 1, abort_flag, p.status, p.wait_limit);
        if (ok) ok = spin_wait(&full_v[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, j, st);
        if (j == 0 && plo_in_k) tc_commit(&empty_k[0]);
        if (more) {
          ok = spin_wait(&full_k[st1], ((j + 1) / NST) & 1, abort_flag, p.status, p.wait_limit);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, st1);
          if (!has_b) tc_commit(&empty_k[st1]);
        }
        if (has_b) {
          ok = spin_wait(&p_full[1], j & 1, abort_flag, p.status, p.wait_limit);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, j, st);
        }
        tc_commit(&empty_v[st]);
        if (has_b && more) {
          issue_s(1, st1);
          tc_commit(&empty_k[st1]);
        }
      }
      tc_commit(fin);
      drain_wait(fin, 0);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax warps
    const int x = warp >> 2;                       // tile
    const int r = tid & 127;                       // row = TMEM lane
    const int tok_local = r >> p.g_shift;
    const int g = r & (G - 1);
    const bool row_valid = (x * TQ + tok_local) < it.q_ntok && (x == 0 || has_b);
    const int qi = it.q_tok0 + x * TQ + tok_local;
    const int64_t qrow = (int64_t(rq.qo_start) + qi) * p.Hq + int64_t(it.kv_head) * G + g;
    int row_end = p.causal ? (rq.kv_len - rq.qo_len + qi + 1) : rq.kv_len;
    row_end = min(row_end, it.kv_tok1);
    if (!row_valid) row_end = 0;
    const float sl2 = p.scale_log2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + x * 128;
    const uint32_t o_col = tmem + lane_base + C::O_COL + x * 128;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = (x == 0) || has_b;

    // One key tile of the online softmax; the first tile of the item (the
    // only one where P may be split into hi + lo) is a separate instance, so
    // that the loop over the others carries only the common path (with both
    // in the loop body the row's registers spilled on every tile).
    auto tile = [&](int j, auto first_tag) -> bool {
      const int k0 = it.kv_tok0 + j * kKvTile;
      ok = warp_wait(&s_full[x], j & 1, abort_flag, p.status, p.wait_limit);
      if (!ok) return false;
      tc_fence_after();
      const int lim = row_end - k0;

      // the whole S row in registers: four loads, one wait
      uint32_t s[128];
      tmem_ld32(s_col + 0, *reinterpret_cast<uint32_t(*)[32]>(s + 0));
      tmem_ld32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
      tmem_ld32(s_col + 64, *reinterpret_cast<uint32_t(*)[32]>(s + 64));
      tmem_ld32(s_col + 96, *reinterpret_cast<uint32_t(*)[32]>(s + 96));
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 128; ++i) asm volatile("" : "+r"(s[i]));
      if (lim < kKvTile) {  // mask past the row's end (diagonal / tail tiles only)
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= lim) s[i] = __float_as_uint(-INFINITY);
      }
      // row max as a tree of three-input maxima: 128 -> 43 -> 15 -> 5 -> 1
      float m43[43];
#pragma unroll
      for (int u = 0; u < 42; ++u)
        m43[u] = fmax3(__uint_as_float(s[3 * u]), __uint_as_float(s[3 * u + 1]), __uint_as_float(s[3 * u + 2]));
      m43[42] = fmaxf(__uint_as_float(s[126]), __uint_as_float(s[127]));
      float m15[15];
#pragma unroll
      for (int u = 0; u < 14; ++u) m15[u] = fmax3(m43[3 * u], m43[3 * u + 1], m43[3 * u + 2]);
      m15[14] = m43[42];
      float m5[5];
#pragma unroll
      for (int u = 0; u < 5; ++u) m5[u] = fmax3(m15[3 * u], m15[3 * u + 1], m15[3 * u + 2]);
      const float mx2 = fmax3(fmax3(m5[0], m5[1], m5[2]), m5[3], m5[4]) * sl2;
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

      constexpr bool kFirstTile = decltype(first_tag)::value;
      const bool lo_split = kFirstTile && lo_split0;
      if (lo_split && x == 0 && C::OFF_PLO_A == C::OFF_K && has_b) {
        // tile A's P_lo reuses K stage 0: S_B(0) must be done reading it
        ok = warp_wait(&s_full[1], 0, abort_flag, p.status, p.wait_limit);
        if (!ok) return false;
      }

      // p = exp2(s * scale_log2 - m), row sum, P (hi) into TMEM over S.  The
      // row sum runs in two independent chains (one long chain of dependent
      // adds would set the pace; more chains cost registers).  The first key
      // tile of a sequence is compiled apart: only there may P be split into
      // hi + lo.  (Measured slower and left out: a quarter or more of the
      // exponentials on the FMA pipe by a polynomial, and exponentials
      // against the running maximum with the tile maximum taken alongside.)
      const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m_use, -m_use);
      auto softmax_p = [&](auto first_tag) -> float {
        constexpr bool kFirst = decltype(first_tag)::value;
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ph[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t lw[4];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int i = 4 * u + v, k = 32 * c + 2 * i;
              const float2 t2 =
                  __ffma2_rn(make_float2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])), sc2, nm2);
              const float a = ex2(t2.x), b = ex2(t2.y);
              acc[u & 1] = __fadd2_rn(acc[u & 1], make_float2(a, b));
              ph[i] = Elt<T>::from_f2(a, b);
              if (kFirst && lo_split) {
                const float2 hi = Elt<T>::to_f2(ph[i]);
                lw[v] = Elt<T>::from_f2(a - hi.x, b - hi.y);
              }
            }
            if (kFirst && lo_split) {
              // keys 32c + 8u .. +7 of row r -> K-major 128-byte-swizzled smem
              const int cc = (c & 1) * 4 + u;
              *reinterpret_cast<uint4*>(smem + plo_off(x) + (c >> 1) * C::BLK + r * 128 + ((cc ^ (r & 7)) * 16)) =
                  make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
          tmem_st16(s_col + c * 16, ph);
        }
        const float2 sum = __fadd2_rn(acc[0], acc[1]);
        return sum.x + sum.y;
      };
      const float rs = softmax_p(first_tag);
      // PV_x(j-1) is complete here: it was issued before S_x(j), and the
      // commit that completed s_full for S_x(j) tracks every MMA issued
      // before it, so O may be rescaled without a wait of its own
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(o_col + c4 * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(o_col + c4 * 32, o);
        }
      }
      // keys past the end of the range: zero their V rows (they may hold
      // anything, and 0 * NaN would poison O); cp.async already zero-filled
      if (x == 0 && use_tma && j == nkt - 1) {
        const int valid = it.kv_tok1 - k0;
        if (valid < kKvTile) {
          const int st = j % NST;
          ok = warp_wait(&full_v[st], (j / NST) & 1, abort_flag, p.status, p.wait_limit);
          if (!ok) return false;
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
      l_sum = l_sum * alpha + rs;
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[x]);
      return true;
    };
    if (ok && nkt > 0) ok = tile(0, std::true_type{});
    for (int j = 1; ok && j < nkt; ++j) ok = tile(j, std::false_type{});

    // ---------------------------------------------------------------- epilogue
    pdl_wait();  // (long since returned for the producer) before the first global write
    if (ok && (x == 0 || has_b)) ok = warp_wait(&o_done[x], 0, abort_flag, p.status, p.wait_limit);
    pdl_launch();
    if (ok && (x == 0 || has_b)) {
      tc_fence_after();
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const float lse_v = l_sum > 0.f ? (m_use + __log2f(l_sum)) * kLn2 : -INFINITY;
      const bool partial = it.part_row >= 0;
      // O_x columns [32 c, 32 c + 32) of the row, scaled and written out
      auto store_chunk = [&](int c4, const uint32_t (&o)[32]) {
        if (!row_valid) return;
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
          float4* dst =
              reinterpret_cast<float4*>(p.part_o + (int64_t(it.part_row) + x * kQRows + r) * D + c4 * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(o[4 * v + 0]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                 __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
        }
      };
      if constexpr (D <= 128) {
        // the whole O row in registers with one wait, then the stores
        uint32_t o[D / 32][32];
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) tmem_ld32(o_col + c4 * 32, o[c4]);
        tmem_wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4)
#pragma unroll
          for (int i = 0; i < 32; ++i) asm volatile("" : "+r"(o[c4][i]));
        // direct output leaves by TMA stores: O (scaled and packed) is staged
        // in the tile's Q slot, free since the tile's last S MMA, as the
        // 128-byte-swizzled rows that the out maps copy -- a full tile as one
        // 128-row box (the Q load's box), a partial one as the 32-row boxes
        // its valid rows fill, the rows after those copied out of the staged
        // tile row by row; split states are written row by row
        const int vrows = partial ? 0 : min(kQRows, (it.q_ntok - x * TQ) << p.g_shift);
        const int srows = vrows & ~31;  // rows the TMA stores carry
        if (srows > 0) {
          if (r < srows) {
            uint8_t* orow = smem + C::OFF_Q + x * C::Q_BYTES + r * 128;
#pragma unroll
            for (int kb = 0; kb < NKB; ++kb)
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                const int e = kb * 64 + c * 8;  // the chunk's first column
                const uint32_t* v = &o[e >> 5][e & 31];
                uint4 w;
                w.x = Elt<T>::from_f2(__uint_as_float(v[0]) * inv_l, __uint_as_float(v[1]) * inv_l);
                w.y = Elt<T>::from_f2(__uint_as_float(v[2]) * inv_l, __uint_as_float(v[3]) * inv_l);
                w.z = Elt<T>::from_f2(__uint_as_float(v[4]) * inv_l, __uint_as_float(v[5]) * inv_l);
                w.w = Elt<T>::from_f2(__uint_as_float(v[6]) * inv_l, __uint_as_float(v[7]) * inv_l);
                *reinterpret_cast<uint4*>(orow + kb * C::BLK + ((c ^ (r & 7)) << 4)) = w;
              }
          } else {  // the partial tile's last rows, row by row
#pragma unroll
            for (int c4 = 0; c4 < D / 32; ++c4) store_chunk(c4, o[c4]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_st[x]);
          if (r == 0 && mbar_wait(&o_st[x], 0, abort_flag, p.status, p.wait_limit)) {
            const int tok0 = rq.qo_start + it.q_tok0 + x * TQ;
            if (srows == kQRows) {
#pragma unroll
              for (int kb = 0; kb < NKB; ++kb)
                tma_store_3d(&o_map, q_addr(x) + kb * C::BLK, kb * 64, it.kv_head * G, tok0);
            } else {
#pragma unroll
              for (int b = 0; b < 3; ++b)
                if (b < (srows >> 5)) {
#pragma unroll
                  for (int kb = 0; kb < NKB; ++kb)
                    tma_store_3d(&o32_map, q_addr(x) + kb * C::BLK + b * 32 * 128, kb * 64, it.kv_head * G,
                                 tok0 + ((b * 32) >> p.g_shift));
                }
            }
            tma_store_commit();
            tma_store_wait_read();  // the Q slot is read before the CTA's memory goes away
          }
        } else {
#pragma unroll
          for (int c4 = 0; c4 < D / 32; ++c4) store_chunk(c4, o[c4]);
        }
      } else {
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(o_col + c4 * 32, o);
          tmem_wait_ld(o);
          store_chunk(c4, o);
        }
      }
      if (row_valid) {
        if (!partial) {
          if (p.lse) p.lse[qrow] = lse_v;
        } else {
          p.part_lse[it.part_row + x * kQRows + r] = lse_v;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  // a softmax warp that gave up between its P stores and their wait still
  // has TMEM stores in flight: they complete before TMEM is released
  if (warp < C::WARP_PROD) tmem_wait_st();
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <typename T, int D, int NT>
cudaError_t launch_prefill_t(const RunArgs& a, const CUtensorMap* kv_map, const CUtensorMap* q_map,
                             const CUtensorMap* o_map, const KParams& kp, int use_tma) {
  using C = PreCfg<D, NT>;
  // o_map[0]: 128-row boxes over out; o_map[1]: 32-row boxes
  static std::atomic<uint64_t> attr_set{0};
  cudaError_t e = set_smem_once(attr_set, reinterpret_cast<const void*>(prefill_kernel<T, D, NT>), C::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_kernel<T, D, NT>, unsigned(a.hp->n_pre), unsigned(C::THREADS), size_t(C::SMEM), a.stream,
                    *kv_map, *q_map, o_map[0], o_map[1], kp, use_tma);
}

template <typename T>
cudaError_t launch_prefill_dt(const RunArgs& a, const CUtensorMap* kv_map, const CUtensorMap* q_map,
                              const CUtensorMap* o_map, const KParams& kp, int use_tma) {
  const bool one = a.hp->pre_tiles == 1;
  switch (a.hp->D) {
    case 64: return one ? launch_prefill_t<T, 64, 1>(a, kv_map, q_map, o_map, kp, use_tma)
                        : launch_prefill_t<T, 64, 2>(a, kv_map, q_map, o_map, kp, use_tma);
    case 128: return one ? launch_prefill_t<T, 128, 1>(a, kv_map, q_map, o_map, kp, use_tma)
                         : launch_prefill_t<T, 128, 2>(a, kv_map, q_map, o_map, kp, use_tma);
    case 256: return one ? launch_prefill_t<T, 256, 1>(a, kv_map, q_map, o_map, kp, use_tma) : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

KParams make_params(const RunArgs& a);

cudaError_t launch_prefill(const RunArgs& a, const CUtensorMap* map_sw128, const CUtensorMap* map_q,
                           const CUtensorMap* map_o) {
  if (a.hp->n_pre == 0) return cudaSuccess;
  KParams kp = make_params(a);
  kp.n_items = a.hp->n_pre;
  const int use_tma = (map_sw128 != nullptr && !a.force_cp_async && a.hp->ps >= 8) ? 1 : 0;
  CUtensorMap dummy;
  memset(&dummy, 0, sizeof(dummy));
  const CUtensorMap* m = use_tma ? map_sw128 : &dummy;
  return a.hp->dtype == PA_BF16 ? launch_prefill_dt<__nv_bfloat16>(a, m, map_q, map_o, kp, use_tma)
                                 : launch_prefill_dt<__half>(a, m, map_q, map_o, kp, use_tma);
}

}  // namespace pa
