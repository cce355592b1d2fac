"""Plain restatement of the planner's partition rules (TEST INFRASTRUCTURE).

The timing script of the FlashInfer issue "How are prefill and decode kernels
different?" builds "auxiliary data structures" once per batch
(``begin_forward`` on the indptr arrays) into a caller-owned workspace and
then calls ``forward`` many times.  The library's planner does the same: it
turns the CSR page table into a list of work items and a merge map.  This
module states those rules a second time, in Python, so that the metadata the
C++ planner writes can be compared with it bit for bit.

Rules (the planner is deterministic; nothing depends on timing):

1. Per request: qo_b, pages_b, kv_b = (pages_b - 1) * page_size + last_b
   (see ``oracle.attention.kv_len_of``), page_start_b.
2. Small-query requests go to the decode kernels: G = Hq/Hkv is one of
   1, 2, 4, 8, 16, the request's R_b = qo_b * G packed (token, head) rows
   number at most 32, a request with qo_b > 1 has kv_b > 128 (more keys
   than one prefill key tile), and ``force_prefill`` is off.  With
   ``decode_cuda_cores``, or at head_dim 256, only qo_b == 1 at G <= 8
   qualifies.  Every other request with qo_b >= 1 goes to the tensor-core
   prefill kernel.  The decode items run on CUDA cores (header word 29 = 1)
   in those two cases, or when G <= 2 and no small-query request has
   qo_b > 1; else on the warp-MMA kernel (0).  An item's row class is
   0, 1, 2 for R_b <= 8, 16, 32 (class 3, 64 rows, is never planned).
3. Decode split ("kv-parallelism", the split-k of the same issue): with
   P_dec = sum over decode requests of pages_b * Hkv and
   target = 4 * num_sms, the first choice is
   c0 = clamp(ceil(P_dec / target), lo = max(1, 256 // page_size),
   hi = max(1, 2048 // page_size)) pages.  Let N(c) = sum over decode
   requests of Hkv * ceil(pages_b / c), the item count at chunk c.  If
   N(hi) <= 2 * num_sms and 4 * N(hi) >= 3 * num_sms (at chunk hi the items
   fit one wave of resident CTAs and cover at least 3/4 of the SMs), the
   chunk is hi.  Else, if N(c0) > 2 * num_sms (more than one wave) and
   N(hi) <= 2 * num_sms, the chunk is the smallest c with
   N(c) <= 2 * num_sms; else c0 (an override replaces all of these).  Request b is cut into
   n = ceil(pages_b / chunk) splits, split s covering pages
   [floor(s * pages_b / n), floor((s + 1) * pages_b / n)), for every kv head.
4. Prefill items: 256 packed rows = (256 / G) query tokens x G heads (two
   128-row tiles); 128 packed rows (one tile) at head_dim 256, with
   ``prefill_q_tiles`` = 1, or when n1 = sum over prefill requests (and
   cascade prefixes, of T_g tokens over np_g * page_size keys) of
   ceil(qo_b / (128 / G)), n2, the same at 256 / G, and w1 = sum of
   ceil(qo_b / (128 / G)) * ceil(kv_b / 128) satisfy 2 * n1 <= 3 * n2
   (most two-tile items would run only their first tile) and w1 <= 8 * n1
   (their key ranges are short).  Item [t0, t0 + n) of request b needs keys [0, e) with
   e = kv_b - qo_b + t0 + n (causal) or kv_b; that is ceil(e / 128) key
   tiles of 128.  With W = the
   sum of key tiles over all (tile, kv head) items and target = 2 * num_sms,
   the chunk is max(8, ceil(W / target)) key tiles (or the override); an item
   with more key tiles is cut into ceil(tiles / chunk) splits.
5. Partial rows (fp32, in the workspace) are handed out in emission order:
   decode splits first (request, then kv head), then prefill splits (request,
   tile, kv head); a split group of S splits and R rows per split takes S * R
   consecutive rows (R = R_b for decode items).  One merge entry is emitted
   per (query token, kv head) of a split group: {out_row0, part_row0,
   nsplit, split_stride}.
6. Decode items are then ordered by row class, then by decreasing key count;
   prefill items by decreasing key count; ties keep emission order (stable
   sorts).  The hardware's in-order block dispatch so starts the long items
   first, and each row class is one launch over consecutive items; header
   words 33..36 hold the number of decode items of each class.

Metadata layout (int32 words, every region 256-byte aligned), which is what
``pagedattn_debug_plan_dump`` returns and ``pagedattn_plan`` copies to the
start of the workspace:

    header[64]  magic 0x50414731, version 2, B, Hq, Hkv, D, page_size,
                num_pages, dtype, causal, T, nnz, n_dec, n_pre, n_merge,
                n_part_rows, dec_chunk_pages, pre_chunk_tiles, num_sms, G,
                off_pages, off_req, off_dec, off_pre, off_merge, blob_bytes,
                off_part_o, off_part_lse, total_bytes, dec_cuda_cores, 0, 0,
                [32] status word, [33..36] decode items per row class,
                [37] cache layout (0 NHD, 1 HND), [38] shared-prefix groups,
                [39] 128-row query tiles per prefill item, 0...
    pages[nnz]       copy of kv_page_indices
    req[B + groups][4]  qo_start, qo_len, kv_len, page_start (group g's prefix: entry B + g,
                     qo_len 0, its query tokens' qo_start, the prefix pages after the requests')
    dec[n_dec][8]    req, kv_head, tok0, tok1, part_row(-1 = direct), page_start of req, 0, 0
    pre[n_pre][8]    req, kv_head, q_tok0, q_ntok, kv_tok0, kv_tok1, part_row, 0
    merge[n][4]      out_row0, part_row0, nsplit, split_stride
"""
from __future__ import annotations

import numpy as np

from .attention import PlanError, request_lengths

MAGIC = 0x50414731
VERSION = 5
HDR_WORDS = 64
STATUS_WORD = 32
Q_ROWS = 128       # packed query rows per prefill MMA tile (G must divide it)
ITEM_ROWS = 256    # packed query rows per prefill work item
KV_TILE = 128      # keys per prefill key tile
DEC_ITEMS_PER_SM = 4
DEC_WAVE_PER_SM = 2   # resident small-query CTAs per SM
PRE_ITEMS_PER_SM = 2
PRE_MIN_CHUNK_TILES = 8
DECODE_GROUPS = (1, 2, 4, 8, 16)
DEC_MAX_ROWS = 32
DEC_CLASS_ROWS = (8, 16, 32, 64)

FP16, BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED = 0, 1, 2


class Unsupported(ValueError):
    pass


def _cdiv(a, b):
    return -(-a // b)


def _align(x, a=256):
    return _cdiv(x, a) * a


def build(qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, num_qo_heads,
          num_kv_heads, head_dim, page_size, num_pages, dtype=BF16, causal=True, num_sms=148,
          force_prefill=False, decode_chunk_pages=0, prefill_chunk_tiles=0, decode_cuda_cores=False,
          kv_layout="NHD", prefix_groups=None, prefill_q_tiles=0):
    """Return the metadata blob (np.int32) the planner must produce.
    ``prefix_groups`` = (group_indptr, prefix_page_indptr, prefix_page_indices)
    plans a shared-prefix cascade (rule 7)."""
    Hq, Hkv, D, ps = int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size)
    if Hq < 1 or Hkv < 1 or Hq % Hkv:
        raise PlanError("num_qo_heads must be a positive multiple of num_kv_heads")
    G = Hq // Hkv
    if D not in (64, 128, 256):
        raise Unsupported("head_dim")
    if ps < 1 or ps > 128 or (ps & (ps - 1)):
        raise Unsupported("page_size")
    if dtype not in (FP16, BF16):
        raise Unsupported("dtype")
    if Q_ROWS % G:
        raise Unsupported("group size must divide 128")
    if num_sms < 1:
        raise PlanError("num_sms")
    lens = request_lengths(qo_indptr, kv_page_indptr, kv_last_page_len, ps)
    B = len(lens)
    indices = np.asarray(kv_page_indices, np.int64)
    nnz = int(np.asarray(kv_page_indptr)[-1])
    if len(indices) < nnz:
        raise PlanError("kv_page_indices shorter than kv_page_indptr[B]")
    indices = indices[:nnz]
    if nnz and (indices.min() < 0 or indices.max() >= num_pages):
        raise PlanError("page id out of range")
    for (qo, kv, _, _) in lens:
        if qo > 0 and (kv < 1 or (causal and qo > kv)):
            raise PlanError("query rows without keys")
    T = int(np.asarray(qo_indptr)[-1])

    # -- rule 7: shared-prefix groups: requests r0..r1-1, T_g query tokens,
    # prefix of np_g full pages stored after the requests' pages
    groups, grp_of, tok_off, pindices = [], [-1] * B, [0] * B, np.zeros(0, np.int64)
    if prefix_groups is not None:
        gind, pind = (np.asarray(x, np.int64) for x in prefix_groups[:2])
        pindices = np.asarray(prefix_groups[2], np.int64)[:int(pind[-1])]
        if gind[0] != 0 or gind[-1] != B or pind[0] != 0:
            raise PlanError("group_indptr must run from 0 to batch_size")
        if len(pindices) and (pindices.min() < 0 or pindices.max() >= num_pages):
            raise PlanError("prefix page id out of range")
        for g in range(len(gind) - 1):
            r0, r1 = int(gind[g]), int(gind[g + 1])
            npp = int(pind[g + 1] - pind[g])
            groups.append((r0, r1, int(qo_indptr[r1]) - int(qo_indptr[r0]), npp, nnz + int(pind[g])))
            if npp > 0:
                for b in range(r0, r1):
                    grp_of[b] = g
                    tok_off[b] = int(qo_indptr[b]) - int(qo_indptr[r0])
    NG = len(groups)

    is_dec = []
    for (qo, kv, _, _) in lens:
        d = (qo >= 1 and G in DECODE_GROUPS and not force_prefill and qo * G <= DEC_MAX_ROWS
             and (qo == 1 or kv > KV_TILE))
        if decode_cuda_cores or D == 256:
            d = d and qo == 1 and G <= 8
        is_dec.append(d)
    multi = any(d and l[0] > 1 for l, d in zip(lens, is_dec))
    dec_cores = 1 if (decode_cuda_cores or D == 256 or (G <= 2 and not multi)) else 0

    # -- decode items (rule 3)
    p_dec = sum(l[3] * Hkv for l, d in zip(lens, is_dec) if d)
    lo, hi = max(1, 256 // ps), max(1, 2048 // ps)
    chunk = decode_chunk_pages if decode_chunk_pages > 0 else min(max(_cdiv(p_dec, DEC_ITEMS_PER_SM * num_sms), lo), hi)
    if decode_chunk_pages <= 0 and p_dec > 0:
        wave = DEC_WAVE_PER_SM * num_sms

        def n_items(c):
            return sum(Hkv * _cdiv(l[3], c) for l, d in zip(lens, is_dec) if d)

        if n_items(hi) <= wave and 4 * n_items(hi) >= 3 * num_sms:
            chunk = hi
        elif n_items(chunk) > wave and n_items(hi) <= wave:
            chunk = next(c for c in range(chunk, hi + 1) if n_items(c) <= wave)
    part = 0
    dec, merges = [], []
    for b, ((qo, kv, p0, npg), d) in enumerate(zip(lens, is_dec)):
        if not d or grp_of[b] >= 0:
            continue
        ns = _cdiv(npg, chunk)
        R = qo * G
        cls = next(c for c, rows in enumerate(DEC_CLASS_ROWS) if R <= rows)
        qs = int(qo_indptr[b])
        for h in range(Hkv):
            base = part if ns > 1 else -1
            if ns > 1:
                part += ns * R
                for t in range(qo):
                    merges.append(((qs + t) * Hq + h * G, base + t * G, ns, R))
            for s in range(ns):
                t0 = (s * npg // ns) * ps
                t1 = min(((s + 1) * npg // ns) * ps, kv)
                dec.append((b, h, t0, t1, base + s * R if ns > 1 else -1, -1, 0, cls))

    # -- prefill items (rule 4)
    if D == 256:
        pre_tiles = 1
    elif prefill_q_tiles:
        pre_tiles = int(prefill_q_tiles)
    else:   # one tile when most two-tile items would run only their first tile
        qk = [(l[0], l[1]) for l, d in zip(lens, is_dec) if not d and l[0] > 0]
        qk += [(g[2], g[3] * ps) for g in groups if g[3] > 0 and g[2] > 0]
        n1 = sum(_cdiv(q, Q_ROWS // G) for q, _ in qk)
        n2 = sum(_cdiv(q, ITEM_ROWS // G) for q, _ in qk)
        w1 = sum(_cdiv(q, Q_ROWS // G) * _cdiv(k, KV_TILE) for q, k in qk)
        pre_tiles = 1 if (2 * n1 <= 3 * n2 and w1 <= 8 * n1) else 2
    tq = pre_tiles * Q_ROWS // G

    def tiles_of(b):
        qo, kv = lens[b][0], lens[b][1]
        return [(b, t0, min(tq, qo - t0), (kv - qo + t0 + min(tq, qo - t0)) if causal else kv)
                for t0 in range(0, qo, tq)]

    tiles = []  # (b, t0, n, e)
    for b, ((qo, kv, p0, npg), d) in enumerate(zip(lens, is_dec)):
        if d or qo == 0 or grp_of[b] >= 0:
            continue
        tiles += tiles_of(b)
    # cascade: the prefix tiles of virtual request B + g (every key visible),
    # then the group's prefill requests
    gtiles = []
    for g, (r0, r1, Tg, npp, _) in enumerate(groups):
        gt = []
        if npp > 0 and Tg > 0:
            gt = [(B + g, t0, min(tq, Tg - t0), npp * ps) for t0 in range(0, Tg, tq)]
            for b in range(r0, r1):
                if not is_dec[b] and lens[b][0] > 0:
                    gt += tiles_of(b)
        gtiles.append(gt)
    W = sum(_cdiv(e, KV_TILE) for (_, _, _, e) in tiles + [t for gt in gtiles for t in gt]) * Hkv
    ctiles = prefill_chunk_tiles if prefill_chunk_tiles > 0 else max(PRE_MIN_CHUNK_TILES, _cdiv(W, PRE_ITEMS_PER_SM * num_sms))
    pre = []
    for (b, t0, n, e) in tiles:
        nt = _cdiv(e, KV_TILE)
        ns = _cdiv(nt, ctiles)
        qs = int(qo_indptr[b])
        for h in range(Hkv):
            base = part if ns > 1 else -1
            if ns > 1:
                part += ns * n * G
                for t in range(n):
                    merges.append(((qs + t0 + t) * Hq + h * G, base + t * G, ns, n * G))
            for s in range(ns):
                k0 = s * ctiles * KV_TILE
                k1 = min((s + 1) * ctiles * KV_TILE, e)
                pre.append((b, h, t0, n, k0, k1, base + s * n * G if ns > 1 else -1))

    # -- rule 7: cascade blocks, items and merges, group by group
    def tile_splits(e):
        return _cdiv(_cdiv(e, KV_TILE), ctiles)

    for g, (r0, r1, Tg, npp, _) in enumerate(groups):
        if npp == 0 or Tg == 0:
            continue
        nsp = tile_splits(npp * ps)
        nsmax = 1
        for b in range(r0, r1):
            if is_dec[b]:
                nsmax = max(nsmax, _cdiv(lens[b][3], chunk))
        for (b, t0, n, e) in gtiles[g]:
            if b < B:
                nsmax = max(nsmax, tile_splits(e))
        S, TG = nsp + nsmax, Tg * G
        base = part
        part += Hkv * S * TG

        def row(h, s, tok):
            return base + (h * S + s) * TG + tok * G

        for b in range(r0, r1):
            if not is_dec[b]:
                continue
            qo, kv, p0, npg = lens[b]
            ns = _cdiv(npg, chunk)
            cls = next(c for c, rows in enumerate(DEC_CLASS_ROWS) if qo * G <= rows)
            for h in range(Hkv):
                for s in range(ns):
                    t0 = (s * npg // ns) * ps
                    t1 = min(((s + 1) * npg // ns) * ps, kv)
                    dec.append((b, h, t0, t1, row(h, nsp + s, tok_off[b]), -1, 0, cls))
        for (b, t0, n, e) in gtiles[g]:
            ns = tile_splits(e)
            for h in range(Hkv):
                for s in range(ns):
                    k0 = s * ctiles * KV_TILE
                    k1 = min((s + 1) * ctiles * KV_TILE, e)
                    prow = row(h, s, t0) if b >= B else row(h, nsp + s, tok_off[b] + t0)
                    pre.append((b, h, t0, n, k0, k1, prow))
        for h in range(Hkv):
            for b in range(r0, r1):
                qo, kv, p0, npg = lens[b]
                for i in range(qo):
                    if is_dec[b]:
                        own = _cdiv(npg, chunk)
                    else:
                        t0 = (i // tq) * tq
                        own = tile_splits((kv - qo + min(t0 + tq, qo)) if causal else kv)
                    merges.append(((int(qo_indptr[b]) + i) * Hq + h * G, row(h, 0, tok_off[b] + i), nsp + own, TG))

    # -- longest first, stable (rule 6)
    dec = sorted(dec, key=lambda it: (it[7], -(it[3] - it[2])))
    n_class = [sum(1 for it in dec if it[7] == c) for c in range(len(DEC_CLASS_ROWS))]
    pre = sorted(pre, key=lambda it: -(it[5] - it[4]))

    # -- layout
    off_pages = HDR_WORDS * 4
    nnz_all = nnz + len(pindices)
    off_req = _align(off_pages + 4 * nnz_all)
    off_dec = _align(off_req + 16 * (B + NG))
    off_pre = _align(off_dec + 32 * len(dec))
    off_merge = _align(off_pre + 32 * len(pre))
    blob_bytes = _align(off_merge + 16 * len(merges))
    off_part_o = blob_bytes
    off_part_lse = _align(off_part_o + 4 * D * part)
    total = _align(off_part_lse + 4 * part)
    if total >= 2 ** 31:
        raise Unsupported("metadata and partial states exceed 2 GiB")

    blob = np.zeros(blob_bytes // 4, np.int32)
    hdr = [MAGIC, VERSION, B, Hq, Hkv, D, ps, num_pages, dtype, int(bool(causal)), T, nnz_all,
           len(dec), len(pre), len(merges), part, chunk, ctiles, num_sms, G,
           off_pages, off_req, off_dec, off_pre, off_merge, blob_bytes, off_part_o,
           off_part_lse, total, dec_cores]
    blob[:len(hdr)] = hdr
    blob[33:33 + len(n_class)] = n_class
    blob[37] = {"NHD": 0, "HND": 1}[kv_layout] if isinstance(kv_layout, str) else int(kv_layout)
    blob[38] = NG
    blob[39] = pre_tiles
    blob[off_pages // 4: off_pages // 4 + nnz] = indices
    blob[off_pages // 4 + nnz: off_pages // 4 + nnz_all] = pindices
    req = np.array([(int(qo_indptr[b]), qo, kv, p0) for b, (qo, kv, p0, _) in enumerate(lens)],
                   np.int32).reshape(-1, 4)
    blob[off_req // 4: off_req // 4 + 4 * B] = req.reshape(-1)
    for g, (r0, r1, Tg, npp, pstart) in enumerate(groups):  # virtual prefix requests, qo_len 0
        blob[off_req // 4 + 4 * (B + g): off_req // 4 + 4 * (B + g) + 4] = (int(qo_indptr[r0]), 0, npp * ps, pstart)
    for j, it in enumerate(dec):
        blob[off_dec // 4 + 8 * j: off_dec // 4 + 8 * j + 5] = it[:5]
        blob[off_dec // 4 + 8 * j + 5] = lens[it[0]][2]  # the request's page_start; words 6, 7 stay 0
    for j, it in enumerate(pre):
        blob[off_pre // 4 + 8 * j: off_pre // 4 + 8 * j + 7] = it
    for j, it in enumerate(merges):
        blob[off_merge // 4 + 4 * j: off_merge // 4 + 4 * j + 4] = it
    return blob


def decode_header(blob: np.ndarray) -> dict:
    names = ["magic", "version", "B", "Hq", "Hkv", "D", "page_size", "num_pages", "dtype",
             "causal", "T", "nnz", "n_dec", "n_pre", "n_merge", "n_part_rows", "dec_chunk_pages",
             "pre_chunk_tiles", "num_sms", "G", "off_pages", "off_req", "off_dec", "off_pre",
             "off_merge", "blob_bytes", "off_part_o", "off_part_lse", "total_bytes", "dec_cuda_cores"]
    h = {n: int(blob[i]) for i, n in enumerate(names)}
    h["dec_class_items"] = [int(x) for x in blob[33:33 + len(DEC_CLASS_ROWS)]]
    h["kv_layout"], h["n_groups"], h["pre_tiles"] = int(blob[37]), int(blob[38]), int(blob[39])
    return h


def items(blob: np.ndarray):
    """(decode items [n,8], prefill items [n,8], merge entries [n,4]) views."""
    h = decode_header(blob)
    dec = blob[h["off_dec"] // 4: h["off_dec"] // 4 + 8 * h["n_dec"]].reshape(-1, 8)
    pre = blob[h["off_pre"] // 4: h["off_pre"] // 4 + 8 * h["n_pre"]].reshape(-1, 8)
    mer = blob[h["off_merge"] // 4: h["off_merge"] // 4 + 4 * h["n_merge"]].reshape(-1, 4)
    return dec, pre, mer
