"""Seeded synthetic inputs for batched ragged attention over a paged KV cache.

This module only builds inputs: page tables, query chunks and cache contents.
It holds none of the attention arithmetic, so both the fp64 oracle and the CUDA
library may be fed from it without sharing any of the method.

The five workloads follow the shapes of the three source pages:

* ``tiny``        -- four ragged requests, fp16, head_dim 64, page_size 4.
* ``decode``      -- the decode timing script of the FlashInfer issue "How are
                     prefill and decode kernels different?" (128 requests of
                     1024 keys, 8 query heads on 1 kv head, head_dim 128,
                     page_size 16, contiguous page ids), with the last page
                     full.
* ``ragged``      -- 32 short prompts of 16..200 tokens, the scenario of the
                     llama.cpp discussion "Pad for prefill stage?"; a padded
                     twin pads every prompt to 200 tokens.
* ``prefix``      -- 64 requests that append 30 new tokens to one 200-token
                     system prompt, the case of the vLLM issue "Question about
                     efficient memory sharing (prefix sharing)".
* ``mixed``       -- one 8192-token causal prefill next to 256 decodes with
                     1..8k keys each, the serving mix that the llama.cpp thread
                     describes (big prompts plus 1-token generations).

Every random draw comes from a CPU ``torch.Generator`` with a fixed seed, so a
workload is identical on every machine.  Large tensors are drawn in chunks with
their own derived seeds so that memory stays bounded.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np
import torch

WORKLOAD_NAMES = ("tiny", "decode", "ragged", "prefix", "mixed")
_SEEDS = {name: i for i, name in enumerate(WORKLOAD_NAMES)}


@dataclasses.dataclass
class Workload:
    """One batch: page tables (int32 numpy), query and cache (CPU torch)."""

    name: str
    qo_indptr: np.ndarray          # [B+1] int32
    kv_page_indptr: np.ndarray     # [B+1] int32
    kv_page_indices: np.ndarray    # [nnz] int32
    kv_last_page_len: np.ndarray   # [B] int32
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    dtype: torch.dtype
    causal: bool
    q: torch.Tensor                # [T, Hq, D] dtype (CPU)
    kv_cache: torch.Tensor         # [P, 2, page_size, Hkv, D] dtype (CPU)
    gen_kv_lens: Optional[np.ndarray] = None  # the key counts the generator drew

    @property
    def batch_size(self) -> int:
        return int(self.qo_indptr.shape[0] - 1)

    @property
    def total_qo(self) -> int:
        return int(self.qo_indptr[-1])

    def qo_lens(self) -> np.ndarray:
        return np.diff(self.qo_indptr).astype(np.int64)

    def plan_args(self) -> dict:
        return dict(
            qo_indptr=self.qo_indptr,
            kv_page_indptr=self.kv_page_indptr,
            kv_page_indices=self.kv_page_indices,
            kv_last_page_len=self.kv_last_page_len,
            num_qo_heads=self.num_qo_heads,
            num_kv_heads=self.num_kv_heads,
            head_dim=self.head_dim,
            page_size=self.page_size,
            num_pages=self.num_pages,
            causal=self.causal,
        )


# --------------------------------------------------------------------------
# random draws


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def randn(shape, dtype: torch.dtype, seed: int, chunk_rows: int = 1024) -> torch.Tensor:
    """fp32 N(0,1) draws rounded to ``dtype``; the leading dim is drawn in
    chunks of ``chunk_rows`` rows, chunk c from seed ``seed * 1_000_003 + c``."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=dtype)
    if shape[0] == 0:
        return out
    for c, r0 in enumerate(range(0, shape[0], chunk_rows)):
        r1 = min(shape[0], r0 + chunk_rows)
        g = _gen(seed * 1_000_003 + c)
        out[r0:r1] = torch.randn((r1 - r0,) + shape[1:], generator=g, dtype=torch.float32).to(dtype)
    return out


def randperm(n: int, seed: int) -> np.ndarray:
    return torch.randperm(n, generator=_gen(seed)).numpy().astype(np.int32)


def randint_incl(lo: int, hi: int, n: int, seed: int) -> np.ndarray:
    """n integers uniform on the closed range [lo, hi]."""
    return torch.randint(lo, hi + 1, (n,), generator=_gen(seed)).numpy().astype(np.int64)


# --------------------------------------------------------------------------
# page tables


def last_page_len(kv_len: int, page_size: int) -> int:
    """Slots used in the last page of a request holding ``kv_len`` >= 1 keys:
    always in [1, page_size] (a full last page counts page_size, not 0)."""
    return (kv_len - 1) % page_size + 1


def pages_for(kv_len: int, page_size: int) -> int:
    return (kv_len + page_size - 1) // page_size


def build_tables(qo_lens, kv_lens, page_size, physical_of_logical):
    """CSR tables for requests whose pages are numbered consecutively in
    logical order and then renamed through ``physical_of_logical``."""
    qo_lens = [int(x) for x in qo_lens]
    kv_lens = [int(x) for x in kv_lens]
    B = len(qo_lens)
    qo_indptr = np.zeros(B + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo_lens)
    npages = [pages_for(k, page_size) for k in kv_lens]
    kv_page_indptr = np.zeros(B + 1, np.int32)
    kv_page_indptr[1:] = np.cumsum(npages)
    nnz = int(kv_page_indptr[-1])
    logical = np.arange(nnz, dtype=np.int64)
    kv_page_indices = np.asarray(physical_of_logical, np.int64)[logical].astype(np.int32)
    kv_last = np.array([last_page_len(k, page_size) if k > 0 else 1 for k in kv_lens], np.int32)
    return qo_indptr, kv_page_indptr, kv_page_indices, kv_last


def make_custom(name, qo_lens, kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size,
                dtype=torch.float16, causal=True, seed=1234, permute_pages=True,
                extra_pages=0) -> Workload:
    """A random batch of arbitrary lengths (for tests at small sizes)."""
    npages = sum(pages_for(int(k), page_size) for k in kv_lens)
    P = npages + int(extra_pages)
    perm = randperm(P, seed + 1) if permute_pages else np.arange(P, dtype=np.int32)
    tabs = build_tables(qo_lens, kv_lens, page_size, perm[:npages])
    T = int(sum(int(x) for x in qo_lens))
    q = randn((T, num_qo_heads, head_dim), dtype, seed + 2)
    kv = randn((P, 2, page_size, num_kv_heads, head_dim), dtype, seed + 3)
    return Workload(name, *tabs, num_qo_heads, num_kv_heads, head_dim, page_size, P,
                    dtype, causal, q, kv, np.asarray(kv_lens, np.int64))


# --------------------------------------------------------------------------
# the five workloads


def tiny() -> Workload:
    """4 requests, qo {1,3,5,8}, kv {8,13,17,24}, 2 qo heads on 1 kv head,
    head_dim 64, page_size 4, fp16, physical pages a random permutation."""
    s = _SEEDS["tiny"]
    qo, kv, ps = [1, 3, 5, 8], [8, 13, 17, 24], 4
    n = sum(pages_for(k, ps) for k in kv)  # 2+4+5+6 = 17
    perm = randperm(n, s * 100 + 1)
    tabs = build_tables(qo, kv, ps, perm)
    q = randn((sum(qo), 2, 64), torch.float16, s * 100 + 2)
    cache = randn((n, 2, ps, 1, 64), torch.float16, s * 100 + 3)
    return Workload("tiny", *tabs, 2, 1, 64, ps, n, torch.float16, True, q, cache,
                    np.asarray(kv, np.int64))


def decode(batch_size: int = 128, seq_len: int = 1024, num_qo_heads: int = 8) -> Workload:
    """The decode script's batch: ``batch_size`` requests, 1 query token
    each, ``seq_len`` keys, Hq 8 / Hkv 1, head_dim 128, page_size 16, page ids
    0..P-1 in order (each request owns a contiguous run of 64 pages).
    ``num_qo_heads`` re-heads it (profiling other group sizes)."""
    s = _SEEDS["decode"]
    ps, Hq, Hkv, D = 16, int(num_qo_heads), 1, 128
    pages_per_seq = pages_for(seq_len, ps)
    P = pages_per_seq * batch_size
    tabs = build_tables([1] * batch_size, [seq_len] * batch_size, ps, np.arange(P, dtype=np.int32))
    q = randn((batch_size, Hq, D), torch.float16, s * 100 + 2)
    cache = randn((P, 2, ps, Hkv, D), torch.float16, s * 100 + 3)
    return Workload("decode", *tabs, Hq, Hkv, D, ps, P, torch.float16, True, q, cache,
                    np.full(batch_size, seq_len, np.int64))


def ragged(padded: bool = False, batch_size: int = 32) -> Workload:
    """32 prompts with lengths uniform on [16, 200], qo_len = kv_len, causal,
    Hq 32 / Hkv 8, head_dim 128, page_size 16, bf16, shuffled page ids.

    The padded twin holds the same cache and page ids, with every request
    extended to 200 tokens (13 pages).  The unpadded batch uses the first
    ceil(L/16) pages of each request, and its queries are the first L query
    rows of the padded request, so the real rows of both runs see the same
    keys and values."""
    s = _SEEDS["ragged"]
    ps, Hq, Hkv, D, Lmax = 16, 32, 8, 128, 200
    lens = randint_incl(16, Lmax, batch_size, s * 100 + 1)
    pp = pages_for(Lmax, ps)
    P = pp * batch_size
    perm = randperm(P, s * 100 + 4)
    qpad = randn((batch_size * Lmax, Hq, D), torch.bfloat16, s * 100 + 2)
    cache = randn((P, 2, ps, Hkv, D), torch.bfloat16, s * 100 + 3)
    if padded:
        tabs = build_tables([Lmax] * batch_size, [Lmax] * batch_size, ps, perm)
        return Workload("ragged_padded", *tabs, Hq, Hkv, D, ps, P, torch.bfloat16, True, qpad, cache,
                        np.full(batch_size, Lmax, np.int64))
    qo_indptr = np.zeros(batch_size + 1, np.int32)
    qo_indptr[1:] = np.cumsum(lens)
    kv_page_indptr = np.zeros(batch_size + 1, np.int32)
    idx: List[int] = []
    rows = []
    for b, L in enumerate(lens):
        n = pages_for(int(L), ps)
        idx.extend(perm[b * pp: b * pp + n].tolist())
        kv_page_indptr[b + 1] = kv_page_indptr[b] + n
        rows.append(qpad[b * Lmax: b * Lmax + int(L)])
    last = np.array([last_page_len(int(L), ps) for L in lens], np.int32)
    q = torch.cat(rows, 0).contiguous()
    return Workload("ragged", qo_indptr, kv_page_indptr, np.array(idx, np.int32), last,
                    Hq, Hkv, D, ps, P, torch.bfloat16, True, q, cache, lens.astype(np.int64))


def prefix(duplicated: bool = False, batch_size: int = 64) -> Workload:
    """64 requests = one 200-token prefix + 30 own tokens (qo 30, kv 230),
    Hq 32 / Hkv 8, head_dim 128, page_size 16, bf16.

    A 200-token prefix fills 12 pages and 8 slots of a 13th.  Only the last
    page of a request may be partial, so the 12 full pages are shared by all
    page tables, and the 13th page is per request: slots 0..7 repeat the
    prefix tokens 192..199, slots 8..15 hold the request's tokens 200..207.
    Two private pages (16 + 6 tokens) follow: 15 pages per request, last 6,
    12 + 3*64 = 204 physical pages.

    ``duplicated=True`` gives every request its own copy of the 12 shared
    pages (same values), the memory layout without sharing."""
    s = _SEEDS["prefix"]
    ps, Hq, Hkv, D = 16, 32, 8, 128
    shared, own = 12, 3
    P_shared = shared + own * batch_size
    base = randn((P_shared, 2, ps, Hkv, D), torch.bfloat16, s * 100 + 3)
    # the 8 prefix rows that open every request's 13th page are one copy
    pre_tail = randn((1, 2, 8, Hkv, D), torch.bfloat16, s * 100 + 5)[0]
    for b in range(batch_size):
        base[shared + own * b, :, :8] = pre_tail
    perm = randperm(P_shared, s * 100 + 4)  # physical id of each logical page
    if duplicated:
        P = batch_size * (shared + own)
        cache = torch.empty((P, 2, ps, Hkv, D), dtype=torch.bfloat16)
        idx = []
        for b in range(batch_size):
            for j in range(shared):
                pid = b * (shared + own) + j
                cache[pid] = base[j]
                idx.append(pid)
            for j in range(own):
                pid = b * (shared + own) + shared + j
                cache[pid] = base[shared + own * b + j]
                idx.append(pid)
    else:
        P = P_shared
        cache = torch.empty_like(base)
        cache[torch.from_numpy(perm.astype(np.int64))] = base
        idx = []
        for b in range(batch_size):
            idx.extend(perm[:shared].tolist())
            idx.extend(perm[shared + own * b: shared + own * (b + 1)].tolist())
    qo_indptr = np.arange(0, 30 * batch_size + 1, 30, dtype=np.int32)
    kv_page_indptr = np.arange(0, 15 * batch_size + 1, 15, dtype=np.int32)
    last = np.full(batch_size, 6, np.int32)
    q = randn((30 * batch_size, Hq, D), torch.bfloat16, s * 100 + 2)
    name = "prefix_duplicated" if duplicated else "prefix"
    return Workload(name, qo_indptr, kv_page_indptr, np.array(idx, np.int32), last,
                    Hq, Hkv, D, ps, P, torch.bfloat16, True, q, cache,
                    np.full(batch_size, 230, np.int64))


def mixed(num_decode: int = 256, prefill_len: int = 8192, kv_lo: int = 512, kv_hi: int = 8192,
          num_qo_heads: int = 64, num_kv_heads: int = 8, decode_qo: int = 1) -> Workload:
    """One causal prefill of ``prefill_len`` tokens (request 0; none when 0)
    next to ``num_decode`` decodes of ``decode_qo`` query tokens each
    (speculative-decoding shapes when > 1) with kv_len uniform on
    [kv_lo, kv_hi]; Hq 64 / Hkv 8, head_dim 128, page_size 16, bf16, random
    page ids."""
    s = _SEEDS["mixed"]
    ps, D = 16, 128
    kvd = randint_incl(kv_lo, kv_hi, num_decode, s * 100 + 1)
    pre = [prefill_len] if prefill_len > 0 else []
    qo = pre + [int(decode_qo)] * num_decode
    kv = pre + [int(x) for x in kvd]
    n = sum(pages_for(k, ps) for k in kv)
    perm = randperm(n, s * 100 + 4)
    tabs = build_tables(qo, kv, ps, perm)
    q = randn((sum(qo), num_qo_heads, D), torch.bfloat16, s * 100 + 2)
    cache = randn((n, 2, ps, num_kv_heads, D), torch.bfloat16, s * 100 + 3, chunk_rows=512)
    return Workload("mixed", *tabs, num_qo_heads, num_kv_heads, D, ps, n, torch.bfloat16, True, q, cache,
                    np.asarray(kv, np.int64))


def split_prefix(w: Workload, group_indptr, prefix_pages):
    """Re-express a batch whose requests in each group begin with the same
    full pages as a shared-prefix cascade: returns (prefix_groups, plan
    arguments for the requests' own pages).  prefix_pages[g] pages are taken
    off the front of every page list of group g (they must be identical)."""
    gind = np.asarray(group_indptr, np.int64)
    own_lists, pre_ind, pre_ptr = [], [], [0]
    for g in range(len(gind) - 1):
        k = int(prefix_pages[g])
        lists = [w.kv_page_indices[w.kv_page_indptr[b]:w.kv_page_indptr[b + 1]] for b in range(gind[g], gind[g + 1])]
        if k:
            head = lists[0][:k]
            assert all(np.array_equal(l[:k], head) for l in lists), "group pages differ"
            pre_ind += [int(x) for x in head]
        pre_ptr.append(len(pre_ind))
        own_lists += [l[k:] for l in lists]
    own_ptr = np.zeros(len(own_lists) + 1, np.int32)
    own_ptr[1:] = np.cumsum([len(l) for l in own_lists])
    own_ind = np.concatenate(own_lists).astype(np.int32) if own_lists else np.zeros(0, np.int32)
    args = w.plan_args()
    args.update(kv_page_indptr=own_ptr, kv_page_indices=own_ind)
    groups = (np.asarray(gind, np.int32), np.asarray(pre_ptr, np.int32), np.asarray(pre_ind, np.int32))
    return groups, args


def prefix_decode(batch_size: int = 64, prefix_len: int = 4096, own_lo: int = 100, own_hi: int = 500,
                  num_qo_heads: int = 32, num_kv_heads: int = 8) -> Workload:
    """``batch_size`` one-token decodes that all continue one ``prefix_len``-
    token prompt (whole pages, physically shared: the same page ids open
    every page list) followed by U[own_lo, own_hi] tokens of their own;
    head_dim 128, page_size 16, bf16."""
    s = _SEEDS["prefix"] * 100 + 50
    ps, D = 16, 128
    assert prefix_len % ps == 0
    own = randint_incl(own_lo, own_hi, batch_size, s + 1)
    shared = prefix_len // ps
    own_pages = [pages_for(int(k), ps) for k in own]
    n = shared + sum(own_pages)
    perm = randperm(n, s + 2)
    lists, nxt = [], shared
    for np_b in own_pages:
        lists.append(np.concatenate([perm[:shared], perm[nxt:nxt + np_b]]))
        nxt += np_b
    kv = [prefix_len + int(k) for k in own]
    qo = [1] * batch_size
    qo_indptr = np.zeros(batch_size + 1, np.int32)
    qo_indptr[1:] = np.cumsum(qo)
    kv_page_indptr = np.zeros(batch_size + 1, np.int32)
    kv_page_indptr[1:] = np.cumsum([len(l) for l in lists])
    kv_page_indices = np.concatenate(lists).astype(np.int32)
    kv_last = np.array([last_page_len(k, ps) for k in kv], np.int32)
    q = randn((batch_size, num_qo_heads, D), torch.bfloat16, s + 3)
    cache = randn((n, 2, ps, num_kv_heads, D), torch.bfloat16, s + 4, chunk_rows=512)
    return Workload("prefix_decode", qo_indptr, kv_page_indptr, kv_page_indices, kv_last, num_qo_heads,
                    num_kv_heads, D, ps, n, torch.bfloat16, True, q, cache, np.asarray(kv, np.int64))


def by_name(name: str, **kw) -> Workload:
    return {"tiny": tiny, "decode": decode, "ragged": ragged, "prefix": prefix, "mixed": mixed}[name](**kw)

