// Host planner: validates one batch's page table and cuts it into work items.
//
// The FlashInfer issue "How are prefill and decode kernels different?"
// builds "auxiliary data structures" once per batch (begin_forward on the
// indptr arrays) and reuses them for many forward calls; this is that step.
// Rules (deterministic, no dependence on timing):
//
//  1. Per request b: qo_b = qo_indptr[b+1] - qo_indptr[b], pages_b likewise,
//     kv_b = (pages_b - 1) * page_size + last_b (every page full except the
//     last, 1 <= last <= page_size as the timing script's comment requires).
//  2. Small-query requests go to the decode kernels: with group size
//     G = Hq/Hkv in {1, 2, 4, 8, 16}, a request whose R_b = qo_b * G packed
//     (token, head) rows number at most 32 (one decoded token, or a few
//     speculative ones; at 64 rows the warp-level MMA, not HBM, bounds the
//     small-query kernel, and the tcgen05 prefill kernel ran 64 requests of
//     8 tokens at G 8 in 0.251 ms against 0.401 ms) and, when qo_b > 1, that has more keys than one
//     prefill key tile (kv_b > 128; a shorter one costs the prefill kernel
//     a single key tile), unless force_prefill.  With decode_cuda_cores, or
//     at head_dim 256 (where the warp-MMA kernel's fragments would not fit
//     in registers), only qo_b == 1 at G <= 8 qualifies (the CUDA-core
//     kernel's shapes).  Every other request with rows -> tensor-core
//     prefill.  The decode items run on the CUDA-core kernel in those two
//     cases, or when G <= 2 and every small-query request has qo_b == 1;
//     else on the warp-MMA kernel.  Row class of an item: R_b <= 8, 16 or
//     32 (a fourth class, 64 rows, is never planned).
//  3. Decode split ("kv-parallelism" / split-k in the same issue): chunk c0 =
//     clamp(ceil(P_dec / (4 * SMs)), 256 keys, 2048 keys) in whole pages,
//     P_dec = sum of decode pages x Hkv.  With N(c) = sum over (request,
//     kv head) of ceil(pages_b / c) items, and hi = 2048 keys: if N(hi)
//     fits one wave of 2 * SMs resident CTAs and covers at least 3/4 of the
//     SMs, c = hi (splitting such a batch further only adds split states and
//     a merge: the decode timing script's batch, 128 x 1024 keys, ran 17.5
//     us split in two and 15.9 us whole on a GB300).  Else, if N(c0) exceeds
//     one wave but some c <= hi gives N(c) <= 2 * SMs, the smallest such c is
//     taken (a small batch then runs in one wave).
//     Each (request, kv head) is cut into n = ceil(pages_b / c) splits of
//     floor-spaced page boundaries (split s starts at page
//     floor(s * pages_b / n)), so the splits of a request differ by at most
//     one page.
//  4. Prefill: items of 256 packed rows = 256/G tokens x G heads of one kv
//     head, run as two 128-row MMA tiles that share every K/V tile load (as
//     do the G heads).  Items of one 128-row tile instead (two CTAs then
//     share an SM) at head_dim 256 (two tiles' accumulators would not fit
//     in tensor memory), with prefill_q_tiles = 1, or when most two-tile
//     items would run only their first tile over short key ranges: with
//     n1 = sum over prefill requests (and cascade prefixes) of
//     ceil(qo_b / (128/G)), n2 the same at 256/G and w1 = sum of
//     ceil(qo_b / (128/G)) x ceil(kv_b / 128), when 2 * n1 <= 3 * n2 and
//     w1 <= 8 * n1 (the two-tile CTA has a producer warp for K and one for
//     V, the one-tile CTA one for both, which limits it on long key ranges:
//     64 requests x 8 tokens over 512..8192 keys ran 0.279 ms on one-tile
//     items, 0.251 ms on two-tile items).  An item needs keys [0, kv_b - qo_b + t0 + n) under
//     the bottom-right causal mask; key tiles past that are never visited
//     (the "skips the fully masked out tails" of the llama.cpp discussion
//     "Pad for prefill stage?").  Split when the
//     total key-tile count W exceeds 2 x SMs x chunk: chunk = max(8,
//     ceil(W / (2 * SMs))) key tiles.
//  5. Partial fp32 rows are numbered in emission order (decode splits, then
//     prefill splits); a split group of S splits with R rows each takes S*R
//     consecutive rows; one merge entry per (query token, kv head) of a
//     split group.
//  6. Decode items sorted by row class, then by decreasing key count;
//     prefill items by decreasing key count; ties in emission order.  The
//     in-order block dispatch starts the longest items first, and each row
//     class is one launch over consecutive items.
//  7. Shared-prefix cascade (pagedattn_plan_cascade; the vLLM issue
//     "Question about efficient memory sharing (prefix sharing)" asks to
//     share the computation over a common prompt, not only its memory):
//     the requests of group g, consecutive in the batch, share the full
//     pages prefix_g ahead of their own pages, and every query row sits
//     after that prefix.  The prefix attention of all the group's query
//     tokens (consecutive in q) is one virtual request, index B + g, with
//     no causal mask (its request entry has qo_len 0), planned as prefill
//     items; each real request keeps only its own pages and mask.  Both
//     levels always write partial rows, in one block per (group, kv head):
//     S_g split slots (the prefix's splits first, then room for the most
//     splits any of the group's requests has) of T_g * G rows, token-major,
//     so that every (token, kv head) has its splits at one stride and the
//     merge kernel combines them.  Emission order: everything of the plain
//     requests as above, then group by group its requests' small-query
//     items, its prefix items, its requests' prefill items, its merge
//     entries (kv head, then token).
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "layout.h"

namespace pa {

namespace {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t align256(int64_t x) { return cdiv(x, 256) * 256; }

struct DecTmp { int32_t req, kvh, t0, t1, part, cls; };

// Row class of a small-query item with R packed rows: 0..3 for <= 8, 16, 32, 64.
inline int32_t row_class(int64_t R) { return R <= 8 ? 0 : R <= 16 ? 1 : R <= 32 ? 2 : 3; }
struct PreTmp { int32_t req, kvh, qt0, n, k0, k1, part; };

pagedattn_status fail(std::string* err, pagedattn_status s, const std::string& m) {
  if (err) *err = m;
  return s;
}

}  // namespace

pagedattn_status build_plan(const PlanInputs& in, HostPlan* hp, std::string* err) {
  const int32_t B = in.B, Hq = in.Hq, Hkv = in.Hkv, D = in.D, ps = in.ps;
  if (B < 0) return fail(err, PA_ERR_INVALID_ARG, "batch_size < 0");
  if (Hq < 1 || Hkv < 1 || Hq % Hkv)
    return fail(err, PA_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
  const int32_t G = Hq / Hkv;
  if (D != 64 && D != 128 && D != 256) return fail(err, PA_ERR_UNSUPPORTED, "head_dim must be 64, 128 or 256");
  if (ps < 1 || ps > 128 || (ps & (ps - 1)))
    return fail(err, PA_ERR_UNSUPPORTED, "page_size must be a power of two in [1, 128]");
  if (in.dtype != PA_FP16 && in.dtype != PA_BF16) return fail(err, PA_ERR_UNSUPPORTED, "dtype");
  if (kQRows % G) return fail(err, PA_ERR_UNSUPPORTED, "group size num_qo_heads/num_kv_heads must divide 128");
  if (in.num_sms < 1) return fail(err, PA_ERR_INVALID_ARG, "num_sms < 1");
  if (in.num_pages < 0) return fail(err, PA_ERR_INVALID_ARG, "num_pages < 0");
  if (!in.qo_indptr || !in.kv_page_indptr || (B > 0 && !in.kv_last_page_len))
    return fail(err, PA_ERR_INVALID_ARG, "null host array");
  if (in.qo_indptr[0] != 0 || in.kv_page_indptr[0] != 0)
    return fail(err, PA_ERR_INVALID_ARG, "indptr must start at 0");

  struct Req { int32_t qo, kv, p0, np; };
  std::vector<Req> req(B);
  for (int b = 0; b < B; ++b) {
    const int64_t qo = int64_t(in.qo_indptr[b + 1]) - in.qo_indptr[b];
    const int64_t np = int64_t(in.kv_page_indptr[b + 1]) - in.kv_page_indptr[b];
    if (qo < 0 || np < 0) return fail(err, PA_ERR_INVALID_ARG, "indptr must be nondecreasing");
    const int32_t last = in.kv_last_page_len[b];
    if (np > 0 && (last < 1 || last > ps))
      return fail(err, PA_ERR_INVALID_ARG,
                  "kv_last_page_len[" + std::to_string(b) + "]=" + std::to_string(last) +
                      " outside [1, page_size]");
    const int64_t kv = np > 0 ? (np - 1) * ps + last : 0;
    if (kv > INT32_MAX) return fail(err, PA_ERR_UNSUPPORTED, "kv_len exceeds int32");
    req[b] = {int32_t(qo), int32_t(kv), in.kv_page_indptr[b], int32_t(np)};
  }
  const int64_t nnz = B > 0 ? in.kv_page_indptr[B] : 0;
  if (nnz > 0 && !in.kv_page_indices) return fail(err, PA_ERR_INVALID_ARG, "null kv_page_indices");
  for (int64_t i = 0; i < nnz; ++i) {
    const int32_t p = in.kv_page_indices[i];
    if (p < 0 || p >= in.num_pages)
      return fail(err, PA_ERR_INVALID_ARG,
                  "kv_page_indices[" + std::to_string(i) + "]=" + std::to_string(p) + " out of range");
  }
  for (int b = 0; b < B; ++b) {
    if (req[b].qo > 0 && (req[b].kv < 1 || (in.causal && req[b].qo > req[b].kv)))
      return fail(err, PA_ERR_INVALID_ARG,
                  "request " + std::to_string(b) + " has query rows without keys (qo_len > kv_len)");
  }
  const int32_t T = B > 0 ? in.qo_indptr[B] : 0;

  // -- rule 7: shared-prefix groups (none for a plain plan)
  const int32_t NG = in.n_groups;
  struct Grp { int32_t r0, r1, T, np, p0; };  // requests, query tokens, prefix pages, their offset
  std::vector<Grp> grp(NG > 0 ? NG : 0);
  std::vector<int32_t> grp_of(B, -1), tok_off(B, 0);
  int64_t nnz_pre = 0;
  if (NG < 0) return fail(err, PA_ERR_INVALID_ARG, "num_groups < 0");
  if (NG > 0) {
    if (!in.group_indptr || !in.prefix_page_indptr) return fail(err, PA_ERR_INVALID_ARG, "null group array");
    if (in.group_indptr[0] != 0 || in.group_indptr[NG] != B || in.prefix_page_indptr[0] != 0)
      return fail(err, PA_ERR_INVALID_ARG, "group_indptr must run from 0 to batch_size, prefix_page_indptr from 0");
    nnz_pre = in.prefix_page_indptr[NG];
    if (nnz_pre > 0 && !in.prefix_page_indices) return fail(err, PA_ERR_INVALID_ARG, "null prefix_page_indices");
    for (int g = 0; g < NG; ++g) {
      const int32_t r0 = in.group_indptr[g], r1 = in.group_indptr[g + 1];
      const int32_t np = in.prefix_page_indptr[g + 1] - in.prefix_page_indptr[g];
      if (r1 < r0 || np < 0) return fail(err, PA_ERR_INVALID_ARG, "group indptr arrays must be nondecreasing");
      if (int64_t(np) * ps > INT32_MAX) return fail(err, PA_ERR_UNSUPPORTED, "prefix exceeds int32 keys");
      grp[g] = {r0, r1, in.qo_indptr[r1] - in.qo_indptr[r0], np, int32_t(nnz + in.prefix_page_indptr[g])};
      if (np > 0)
        for (int b = r0; b < r1; ++b) {
          grp_of[b] = g;
          tok_off[b] = in.qo_indptr[b] - in.qo_indptr[r0];
        }
    }
    for (int64_t i = 0; i < nnz_pre; ++i) {
      const int32_t p = in.prefix_page_indices[i];
      if (p < 0 || p >= in.num_pages)
        return fail(err, PA_ERR_INVALID_ARG,
                    "prefix_page_indices[" + std::to_string(i) + "]=" + std::to_string(p) + " out of range");
    }
  }
  const int64_t nnz_all = nnz + nnz_pre;

  const bool dec_group = (G == 1 || G == 2 || G == 4 || G == 8 || G == 16);
  const bool cores_only = in.decode_cuda_cores || D == 256;
  std::vector<char> is_dec(B, 0);
  bool multi_tok = false;
  for (int b = 0; b < B; ++b) {
    const int64_t qo = req[b].qo;
    bool d = qo >= 1 && dec_group && !in.force_prefill && qo * G <= kDecMaxRows && (qo == 1 || req[b].kv > kKvTile);
    if (cores_only) d = d && qo == 1 && G <= 8;
    is_dec[b] = d ? 1 : 0;
    if (d && qo > 1) multi_tok = true;
  }
  const int32_t dec_cores = (cores_only || (G <= 2 && !multi_tok)) ? 1 : 0;

  // -- rule 3: decode items
  int64_t p_dec = 0;
  for (int b = 0; b < B; ++b)
    if (is_dec[b]) p_dec += int64_t(req[b].np) * Hkv;
  const int64_t lo = std::max<int64_t>(1, 256 / ps), hi = std::max<int64_t>(1, 2048 / ps);
  int64_t chunk = in.decode_chunk_pages > 0
                      ? in.decode_chunk_pages
                      : std::min(std::max(cdiv(p_dec, int64_t(4) * in.num_sms), lo), hi);
  if (in.decode_chunk_pages <= 0 && p_dec > 0) {
    const int64_t wave = int64_t(2) * in.num_sms;
    auto items_at = [&](int64_t c) {
      int64_t n = 0;
      for (int b = 0; b < B; ++b)
        if (is_dec[b]) n += cdiv(req[b].np, c) * Hkv;
      return n;
    };
    if (items_at(hi) <= wave && 4 * items_at(hi) >= int64_t(3) * in.num_sms) {
      chunk = hi;
    } else if (items_at(chunk) > wave && items_at(hi) <= wave) {
      int64_t a = chunk, z = hi;  // items_at(a) > wave >= items_at(z); items_at is nonincreasing
      while (z - a > 1) {
        const int64_t mid = (a + z) / 2;
        if (items_at(mid) <= wave) z = mid; else a = mid;
      }
      chunk = z;
    }
  }
  int64_t part = 0;
  std::vector<DecTmp> dec;
  std::vector<MergeEntry> merges;
  for (int b = 0; b < B; ++b) {
    if (!is_dec[b] || grp_of[b] >= 0) continue;
    const int64_t ns = cdiv(req[b].np, chunk);
    const int64_t R = int64_t(req[b].qo) * G;
    const int64_t qs = in.qo_indptr[b];
    for (int h = 0; h < Hkv; ++h) {
      const int64_t base = ns > 1 ? part : -1;
      if (ns > 1) {
        part += ns * R;
        for (int32_t k = 0; k < req[b].qo; ++k)
          merges.push_back({int32_t((qs + k) * Hq + h * G), int32_t(base + int64_t(k) * G), int32_t(ns),
                            int32_t(R)});
      }
      for (int64_t s = 0; s < ns; ++s) {
        const int64_t t0 = (s * req[b].np / ns) * ps;
        const int64_t t1 = std::min<int64_t>(((s + 1) * req[b].np / ns) * ps, req[b].kv);
        dec.push_back({b, h, int32_t(t0), int32_t(t1), ns > 1 ? int32_t(base + s * R) : -1, row_class(R)});
      }
    }
  }

  // -- rule 4: prefill items
  int32_t pre_tiles = 2;
  if (D == 256) {
    pre_tiles = 1;
  } else if (in.prefill_q_tiles > 0) {
    pre_tiles = in.prefill_q_tiles;
  } else {  // one tile when most two-tile items would run only their first tile, over short key ranges
    int64_t n1 = 0, n2 = 0, w1 = 0;
    auto count = [&](int64_t qo, int64_t kv) {
      n1 += cdiv(qo, kQRows / G);
      n2 += cdiv(qo, kItemRows / G);
      w1 += cdiv(qo, kQRows / G) * cdiv(kv, kKvTile);
    };
    for (int b = 0; b < B; ++b)
      if (!is_dec[b] && req[b].qo > 0) count(req[b].qo, req[b].kv);
    for (const Grp& g : grp)
      if (g.np > 0 && g.T > 0) count(g.T, int64_t(g.np) * ps);
    if (2 * n1 <= 3 * n2 && w1 <= 8 * n1) pre_tiles = 1;
  }
  const int32_t tq = pre_tiles * kQRows / G;
  struct Tile { int32_t b, t0, n; int64_t e; };
  auto tiles_of = [&](int b, std::vector<Tile>& out) {
    for (int32_t t0 = 0; t0 < req[b].qo; t0 += tq) {
      const int32_t n = std::min(tq, req[b].qo - t0);
      const int64_t e = in.causal ? int64_t(req[b].kv) - req[b].qo + t0 + n : req[b].kv;
      out.push_back({b, t0, n, e});
    }
  };
  std::vector<Tile> tiles;
  for (int b = 0; b < B; ++b)
    if (!is_dec[b] && req[b].qo > 0 && grp_of[b] < 0) tiles_of(b, tiles);
  // cascade groups: the prefix tiles of virtual request B + g (every key
  // visible), then the group's prefill requests
  std::vector<std::vector<Tile>> gtiles(grp.size());
  for (size_t g = 0; g < grp.size(); ++g) {
    if (grp[g].np == 0 || grp[g].T == 0) continue;
    for (int32_t t0 = 0; t0 < grp[g].T; t0 += tq)
      gtiles[g].push_back({int32_t(B + g), t0, std::min(tq, grp[g].T - t0), int64_t(grp[g].np) * ps});
    for (int b = grp[g].r0; b < grp[g].r1; ++b)
      if (!is_dec[b] && req[b].qo > 0) tiles_of(b, gtiles[g]);
  }
  int64_t W = 0;
  for (auto& t : tiles) W += cdiv(t.e, kKvTile);
  for (auto& gt : gtiles)
    for (auto& t : gt) W += cdiv(t.e, kKvTile);
  W *= Hkv;
  const int64_t ctiles = in.prefill_chunk_tiles > 0 ? in.prefill_chunk_tiles
                                                    : std::max<int64_t>(8, cdiv(W, int64_t(2) * in.num_sms));
  std::vector<PreTmp> pre;
  for (auto& t : tiles) {
    const int64_t nt = cdiv(t.e, kKvTile);
    const int64_t ns = cdiv(nt, ctiles);
    const int64_t qs = in.qo_indptr[t.b];
    for (int h = 0; h < Hkv; ++h) {
      const int64_t base = ns > 1 ? part : -1;
      if (ns > 1) {
        part += ns * t.n * G;
        for (int32_t k = 0; k < t.n; ++k)
          merges.push_back({int32_t((qs + t.t0 + k) * Hq + h * G), int32_t(base + int64_t(k) * G),
                            int32_t(ns), int32_t(t.n * G)});
      }
      for (int64_t s = 0; s < ns; ++s) {
        const int64_t k0 = s * ctiles * kKvTile;
        const int64_t k1 = std::min<int64_t>((s + 1) * ctiles * kKvTile, t.e);
        pre.push_back({t.b, h, t.t0, t.n, int32_t(k0), int32_t(k1),
                       ns > 1 ? int32_t(base + s * int64_t(t.n) * G) : -1});
      }
    }
  }

  // -- rule 7: cascade blocks, items and merges, group by group
  for (size_t g = 0; g < grp.size(); ++g) {
    const Grp& gr = grp[g];
    if (gr.np == 0 || gr.T == 0) continue;
    const int64_t nsp = cdiv(cdiv(int64_t(gr.np) * ps, kKvTile), ctiles);  // prefix splits
    auto tile_splits = [&](const Tile& t) { return cdiv(cdiv(t.e, kKvTile), ctiles); };
    int64_t nsmax = 1;
    for (int b = gr.r0; b < gr.r1; ++b)
      if (is_dec[b]) nsmax = std::max(nsmax, cdiv(req[b].np, chunk));
    for (const Tile& t : gtiles[g])
      if (t.b < B) nsmax = std::max(nsmax, tile_splits(t));
    const int64_t S = nsp + nsmax, TG = int64_t(gr.T) * G;
    const int64_t base = part;
    part += int64_t(Hkv) * S * TG;
    auto row = [&](int h, int64_t s, int64_t tok) { return base + (h * S + s) * TG + tok * G; };
    // the group's small-query requests
    for (int b = gr.r0; b < gr.r1; ++b) {
      if (!is_dec[b]) continue;
      const int64_t ns = cdiv(req[b].np, chunk);
      for (int h = 0; h < Hkv; ++h)
        for (int64_t s2 = 0; s2 < ns; ++s2) {
          const int64_t t0 = (s2 * req[b].np / ns) * ps;
          const int64_t t1 = std::min<int64_t>(((s2 + 1) * req[b].np / ns) * ps, req[b].kv);
          dec.push_back({b, h, int32_t(t0), int32_t(t1), int32_t(row(h, nsp + s2, tok_off[b])),
                         row_class(int64_t(req[b].qo) * G)});
        }
    }
    // the prefix tiles (all tokens of the group), then its prefill requests
    for (const Tile& t : gtiles[g]) {
      const int64_t ns = tile_splits(t);
      const bool prefix = t.b >= B;
      for (int h = 0; h < Hkv; ++h)
        for (int64_t s2 = 0; s2 < ns; ++s2) {
          const int64_t k0 = s2 * ctiles * kKvTile;
          const int64_t k1 = std::min<int64_t>((s2 + 1) * ctiles * kKvTile, t.e);
          const int64_t prow = prefix ? row(h, s2, t.t0) : row(h, nsp + s2, tok_off[t.b] + t.t0);
          pre.push_back({t.b, h, t.t0, t.n, int32_t(k0), int32_t(k1), int32_t(prow)});
        }
    }
    // one merge entry per (kv head, token): the prefix splits then the token's own
    for (int h = 0; h < Hkv; ++h)
      for (int b = gr.r0; b < gr.r1; ++b)
        for (int32_t i = 0; i < req[b].qo; ++i) {
          const int64_t own = is_dec[b] ? cdiv(req[b].np, chunk)
                                        : tile_splits(Tile{b, (i / tq) * tq, 0,
                                                           in.causal ? int64_t(req[b].kv) - req[b].qo +
                                                                           std::min((i / tq + 1) * tq, req[b].qo)
                                                                     : int64_t(req[b].kv)});
          merges.push_back({int32_t((int64_t(in.qo_indptr[b]) + i) * Hq + h * G),
                            int32_t(row(h, 0, tok_off[b] + i)), int32_t(nsp + own), int32_t(TG)});
        }
  }
  if (part > INT32_MAX / 256) return fail(err, PA_ERR_UNSUPPORTED, "too many partial rows");

  // -- rule 6: longest first, stable
  std::stable_sort(dec.begin(), dec.end(), [](const DecTmp& a, const DecTmp& b) {
    if (a.cls != b.cls) return a.cls < b.cls;
    return (a.t1 - a.t0) > (b.t1 - b.t0);
  });
  int32_t n_class[kDecClasses] = {0, 0, 0, 0};
  for (const DecTmp& d : dec) ++n_class[d.cls];
  std::stable_sort(pre.begin(), pre.end(),
                   [](const PreTmp& a, const PreTmp& b) { return (a.k1 - a.k0) > (b.k1 - b.k0); });

  // -- layout
  const int64_t off_pages = HDR_WORDS * 4;
  const int64_t off_req = align256(off_pages + 4 * nnz_all);
  const int64_t off_dec = align256(off_req + 16 * int64_t(B + NG));
  const int64_t off_pre = align256(off_dec + 32 * int64_t(dec.size()));
  const int64_t off_merge = align256(off_pre + 32 * int64_t(pre.size()));
  const int64_t blob_bytes = align256(off_merge + 16 * int64_t(merges.size()));
  const int64_t off_part_o = blob_bytes;
  const int64_t off_part_lse = align256(off_part_o + 4 * int64_t(D) * part);
  const int64_t total = align256(off_part_lse + 4 * part);
  if (total >= (int64_t(1) << 31)) return fail(err, PA_ERR_UNSUPPORTED, "metadata and partial states exceed 2 GiB");

  std::vector<int32_t>& blob = hp->blob;
  blob.assign(size_t(blob_bytes / 4), 0);
  const int32_t hdr[] = {kMagic, kVersion, B, Hq, Hkv, D, ps, in.num_pages, in.dtype, in.causal ? 1 : 0,
                         T, int32_t(nnz_all), int32_t(dec.size()), int32_t(pre.size()), int32_t(merges.size()),
                         int32_t(part), int32_t(chunk), int32_t(ctiles), in.num_sms, G,
                         int32_t(off_pages), int32_t(off_req), int32_t(off_dec), int32_t(off_pre),
                         int32_t(off_merge), int32_t(blob_bytes), int32_t(off_part_o),
                         int32_t(off_part_lse), int32_t(total), dec_cores};
  std::memcpy(blob.data(), hdr, sizeof(hdr));
  for (int c = 0; c < kDecClasses; ++c) blob[H_NDEC_CLASS0 + c] = n_class[c];
  blob[H_LAYOUT] = in.kv_layout;
  blob[H_NGROUPS] = NG;
  blob[H_PRE_TILES] = pre_tiles;
  if (nnz) std::memcpy(blob.data() + off_pages / 4, in.kv_page_indices, size_t(4 * nnz));
  if (nnz_pre) std::memcpy(blob.data() + off_pages / 4 + nnz, in.prefix_page_indices, size_t(4 * nnz_pre));
  for (int b = 0; b < B; ++b) {
    int32_t* r = blob.data() + off_req / 4 + 4 * b;
    r[0] = in.qo_indptr[b];
    r[1] = req[b].qo;
    r[2] = req[b].kv;
    r[3] = req[b].p0;
  }
  for (size_t g = 0; g < grp.size(); ++g) {  // virtual prefix requests: qo_len 0, i.e. every key visible
    int32_t* r = blob.data() + off_req / 4 + 4 * (B + g);
    r[0] = in.qo_indptr[grp[g].r0];
    r[1] = 0;
    r[2] = grp[g].np * ps;
    r[3] = grp[g].p0;
  }
  for (size_t j = 0; j < dec.size(); ++j) {
    int32_t* r = blob.data() + off_dec / 4 + 8 * j;
    r[0] = dec[j].req; r[1] = dec[j].kvh; r[2] = dec[j].t0; r[3] = dec[j].t1; r[4] = dec[j].part;
    r[5] = req[dec[j].req].p0;  // the request's page_start again: one dependent read less for the producer
  }
  for (size_t j = 0; j < pre.size(); ++j) {
    int32_t* r = blob.data() + off_pre / 4 + 8 * j;
    r[0] = pre[j].req; r[1] = pre[j].kvh; r[2] = pre[j].qt0; r[3] = pre[j].n;
    r[4] = pre[j].k0; r[5] = pre[j].k1; r[6] = pre[j].part;
  }
  for (size_t j = 0; j < merges.size(); ++j) {
    int32_t* r = blob.data() + off_merge / 4 + 4 * j;
    r[0] = merges[j].out_row0; r[1] = merges[j].part_row0; r[2] = merges[j].nsplit; r[3] = merges[j].split_stride;
  }

  hp->B = B; hp->Hq = Hq; hp->Hkv = Hkv; hp->D = D; hp->ps = ps; hp->num_pages = in.num_pages;
  hp->dtype = in.dtype; hp->causal = in.causal ? 1 : 0; hp->T = T; hp->nnz = int32_t(nnz_all);
  hp->n_dec = int32_t(dec.size()); hp->n_pre = int32_t(pre.size()); hp->n_merge = int32_t(merges.size());
  hp->n_part = int32_t(part); hp->G = G; hp->num_sms = in.num_sms;
  hp->dec_cores = dec_cores;
  hp->pre_tiles = pre_tiles;
  hp->hnd = in.kv_layout;
  hp->wait_limit_cycles = in.wait_limit_cycles;
  for (int c = 0; c < kDecClasses; ++c) hp->n_dec_class[c] = n_class[c];
  hp->blob_bytes = size_t(blob_bytes); hp->off_part_o = size_t(off_part_o);
  hp->off_part_lse = size_t(off_part_lse); hp->total_bytes = size_t(total);
  hp->off_pages = size_t(off_pages); hp->off_req = size_t(off_req); hp->off_dec = size_t(off_dec);
  hp->off_pre = size_t(off_pre); hp->off_merge = size_t(off_merge);
  hp->kv_len.resize(B);
  for (int b = 0; b < B; ++b) hp->kv_len[b] = req[b].kv;
  return PA_OK;
}

}  // namespace pa
