"""The attention definition, written out plainly in fp64 (TEST INFRASTRUCTURE).

What is computed (sources: FlashInfer issue "How are prefill and decode
kernels different?", the timing script and its API calls; llama.cpp
discussion "Pad for prefill stage?", the reply on skipping masked tails; vLLM
issue "Question about efficient memory sharing (prefix sharing)", the opening
question):

A batch of B requests.  Request b owns ``qo_b`` query rows, packed inside
``q[T, Hq, D]`` between ``qo_indptr[b]`` and ``qo_indptr[b+1]``, and ``kv_b``
keys/values stored in the pages listed by ``kv_page_indices`` between
``kv_page_indptr[b]`` and ``kv_page_indptr[b+1]`` of the cache
``kv_cache[num_pages, 2, page_size, Hkv, D]`` (the "NHD" layout of the timing
script).  Every page of a request is full except the last, which holds
``kv_last_page_len[b]`` slots, 1 <= last <= page_size (the comment beside the
script's ``kv_last_page_len``).

For query row i of request b and query head h, with g = kv head of h:

    n      = number of visible keys (causal: kv_b - qo_b + i + 1)
    s_t    = scale * <q[qo_indptr[b] + i, h, :], K_b[t, g, :]>      t < n
    lse    = ln sum_t exp(s_t)                                     (natural log)
    out    = sum_t exp(s_t - lse) * V_b[t, g, :]

Readings taken where the pages are silent (each is a named helper below, so a
test can swap it for a planted mistake):

* R1 ``visible_keys``: the causal mask is aligned bottom-right -- the new
  query rows are the last ``qo_b`` positions of the request's ``kv_b`` keys
  (prompts appended after a shared prefix; fully masked tails of shorter
  sequences).  qo_b = 1 then sees every key, which is what makes the decode
  output equal the prefill output in the timing script's closing allclose.
* R2 ``K_SLOT``/``V_SLOT``: index 0 of the cache's second dimension is K, 1 is V.
* R3 ``kv_head_of``: consecutive query heads share a kv head (h // (Hq/Hkv)).
* R4 ``lse`` is the natural-log sum of exp of the *scaled* logits.
* R5 ``default_scale``: scale = 1/sqrt(head_dim).
* R6 ``kv_len_of``: kv_b = (pages_b - 1) * page_size + last_b; a last-page
  length of 0 (what the script's ``seq_length % page_size`` gives for 1024
  and 16) violates the script's own 1 <= last <= page_size comment and is
  rejected.

All arithmetic is fp64 on the fp16/bf16 inputs, upcast exactly.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Sequence, Tuple

import numpy as np
import torch

K_SLOT = 0  # R2
V_SLOT = 1  # R2


def default_scale(head_dim: int) -> float:
    """R5: softmax scale 1/sqrt(head_dim)."""
    return 1.0 / math.sqrt(head_dim)


def kv_len_of(num_pages: int, last_page_len: int, page_size: int) -> int:
    """R6: keys held by a request with ``num_pages`` pages whose last page
    holds ``last_page_len`` slots (all earlier pages are full)."""
    if num_pages == 0:
        return 0
    return (num_pages - 1) * page_size + last_page_len


def kv_head_of(h: int, group: int) -> int:
    """R3: the kv head that query head ``h`` reads; ``group`` = Hq / Hkv
    query heads share one kv head (grouped-query attention)."""
    return h // group


def visible_keys(kv_len: int, qo_len: int, i: int, causal: bool) -> int:
    """R1: how many leading keys query row ``i`` (0-based within its request)
    may attend to.  Causal rows sit at absolute positions kv_len - qo_len + i."""
    if not causal:
        return kv_len
    return kv_len - qo_len + i + 1


def locate(pages: Sequence[int], t: int, page_size: int) -> Tuple[int, int]:
    """The physical (page, slot) that holds logical token ``t`` of a request
    whose page list is ``pages`` (the CSR slice of kv_page_indices)."""
    return int(pages[t // page_size]), t % page_size


def softmax_stats(s: np.ndarray) -> Tuple[float, np.ndarray]:
    """lse = ln sum exp(s) (R4) and the normalised weights exp(s - lse),
    evaluated with the max subtracted so that exp never overflows."""
    m = float(np.max(s))
    e = np.exp(s - m)
    z = float(np.sum(e))
    lse = m + math.log(z)
    return lse, np.exp(s - lse)


# ---------------------------------------------------------------------------
# validation (the constraints the pages state, plus the readings above)


class PlanError(ValueError):
    pass


def request_lengths(qo_indptr, kv_page_indptr, kv_last_page_len, page_size):
    """Per-request (qo_len, kv_len, page_start, num_pages), validated."""
    qo_indptr = np.asarray(qo_indptr, np.int64)
    kv_page_indptr = np.asarray(kv_page_indptr, np.int64)
    last = np.asarray(kv_last_page_len, np.int64)
    B = len(qo_indptr) - 1
    if len(kv_page_indptr) != B + 1 or len(last) != B:
        raise PlanError("indptr lengths disagree")
    if qo_indptr[0] != 0 or kv_page_indptr[0] != 0:
        raise PlanError("indptr must start at 0")
    out = []
    for b in range(B):
        qo = int(qo_indptr[b + 1] - qo_indptr[b])
        npg = int(kv_page_indptr[b + 1] - kv_page_indptr[b])
        if qo < 0 or npg < 0:
            raise PlanError("indptr must be nondecreasing")
        if npg > 0 and not (1 <= int(last[b]) <= page_size):
            raise PlanError("last_page_len outside [1, page_size]")
        kv = kv_len_of(npg, int(last[b]), page_size)
        out.append((qo, kv, int(kv_page_indptr[b]), npg))
    return out


def _as_f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().to("cpu").to(torch.float64).numpy()


# ---------------------------------------------------------------------------
# form 1: scalar walk over the page table (tiny inputs only)


def attention_walk(q: torch.Tensor, kv_cache: torch.Tensor, qo_indptr, kv_page_indptr,
                   kv_page_indices, kv_last_page_len, num_qo_heads: int, num_kv_heads: int,
                   head_dim: int, page_size: int, causal: bool = True, sm_scale=None):
    """Loop over every (request, row, head, key); returns fp64 (out, lse)."""
    scale = default_scale(head_dim) if sm_scale is None else float(sm_scale)
    group = num_qo_heads // num_kv_heads
    T = int(np.asarray(qo_indptr)[-1])
    out = np.zeros((T, num_qo_heads, head_dim))
    lse = np.full((T, num_qo_heads), -np.inf)
    qn = _as_f64(q)
    lens = request_lengths(qo_indptr, kv_page_indptr, kv_last_page_len, page_size)
    indices = np.asarray(kv_page_indices, np.int64)
    for b, (qo, kv, p0, npg) in enumerate(lens):
        pages = indices[p0:p0 + npg]
        for i in range(qo):
            row = int(qo_indptr[b]) + i
            n = visible_keys(kv, qo, i, causal)
            if n <= 0:
                raise PlanError("a query row sees no key")
            for h in range(num_qo_heads):
                g = kv_head_of(h, group)
                s = np.empty(n)
                vrows = np.empty((n, head_dim))
                for t in range(n):
                    page, slot = locate(pages, t, page_size)
                    k = kv_cache[page, K_SLOT, slot, g].to(torch.float64).numpy()
                    vrows[t] = kv_cache[page, V_SLOT, slot, g].to(torch.float64).numpy()
                    s[t] = scale * float(np.dot(qn[row, h], k))
                l, w = softmax_stats(s)
                lse[row, h] = l
                acc = np.zeros(head_dim)
                for t in range(n):
                    acc += w[t] * vrows[t]
                out[row, h] = acc
    return out, lse


# ---------------------------------------------------------------------------
# form 2: per (request, kv head) gather of dense K/V, then matmul


def gather_kv(kv_cache: torch.Tensor, pages: np.ndarray, kv_len: int, g: int, page_size: int):
    """Dense fp64 K and V [kv_len, D] of kv head ``g`` for one request."""
    idx = torch.from_numpy(np.asarray(pages, np.int64))
    blk = kv_cache.index_select(0, idx)[:, :, :, g, :]            # [npg, 2, ps, D]
    K = blk[:, K_SLOT].reshape(-1, blk.shape[-1])[:kv_len]
    V = blk[:, V_SLOT].reshape(-1, blk.shape[-1])[:kv_len]
    return _as_f64(K), _as_f64(V)


def _rows_attention(Qr: np.ndarray, K: np.ndarray, V: np.ndarray, nvis: np.ndarray, scale: float):
    """Qr [R, D] rows, row r sees keys [0, nvis[r]).  Returns (out [R,D], lse [R])."""
    S = scale * (Qr @ K.T)                                        # [R, kv]
    cols = np.arange(K.shape[0])[None, :]
    S = np.where(cols < nvis[:, None], S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    Z = E.sum(axis=1, keepdims=True)
    lse = (m + np.log(Z))[:, 0]
    out = (E / Z) @ V
    return out, lse


def attention_gather(q: torch.Tensor, kv_cache: torch.Tensor, qo_indptr, kv_page_indptr,
                     kv_page_indices, kv_last_page_len, num_qo_heads: int, num_kv_heads: int,
                     head_dim: int, page_size: int, causal: bool = True, sm_scale=None):
    """Same definition as ``attention_walk``, vectorised per (request, kv head)."""
    scale = default_scale(head_dim) if sm_scale is None else float(sm_scale)
    group = num_qo_heads // num_kv_heads
    T = int(np.asarray(qo_indptr)[-1])
    out = np.zeros((T, num_qo_heads, head_dim))
    lse = np.full((T, num_qo_heads), -np.inf)
    lens = request_lengths(qo_indptr, kv_page_indptr, kv_last_page_len, page_size)
    indices = np.asarray(kv_page_indices, np.int64)
    for b, (qo, kv, p0, npg) in enumerate(lens):
        if qo == 0:
            continue
        r0 = int(qo_indptr[b])
        nvis = np.array([visible_keys(kv, qo, i, causal) for i in range(qo)], np.int64)
        if nvis.min() <= 0:
            raise PlanError("a query row sees no key")
        for g in range(num_kv_heads):
            K, V = gather_kv(kv_cache, indices[p0:p0 + npg], kv, g, page_size)
            heads = [h for h in range(num_qo_heads) if kv_head_of(h, group) == g]
            for h in heads:
                Qr = _as_f64(q[r0:r0 + qo, h])
                o, l = _rows_attention(Qr, K, V, nvis, scale)
                out[r0:r0 + qo, h] = o
                lse[r0:r0 + qo, h] = l
    return out, lse


def attention(w, form: str = "gather", **kw):
    """Run one form of the oracle on a ``workloads.Workload``."""
    fn = attention_gather if form == "gather" else attention_walk
    return fn(w.q, w.kv_cache, w.qo_indptr, w.kv_page_indptr, w.kv_page_indices,
              w.kv_last_page_len, w.num_qo_heads, w.num_kv_heads, w.head_dim,
              w.page_size, causal=w.causal, **kw)


# ---------------------------------------------------------------------------
# sampled rows (for batches too large to run whole on the CPU)


def request_of_row(qo_indptr, row: int) -> int:
    """The request b whose query rows [qo_indptr[b], qo_indptr[b+1]) hold the
    packed row ``row`` (the CSR query layout of the timing script's
    ``qo_indptr``).  A request with qo_len 0 owns no row, so the answer is
    the last b with qo_indptr[b] <= row."""
    return int(np.searchsorted(np.asarray(qo_indptr), row, side="right") - 1)


def attention_rows(w, rows: Iterable[Tuple[int, int]], sm_scale=None) -> Dict[Tuple[int, int], Tuple[np.ndarray, float]]:
    """fp64 (out[D], lse) for the given (packed query row, query head) pairs.
    Rows of one (request, kv head) share one gather."""
    scale = default_scale(w.head_dim) if sm_scale is None else float(sm_scale)
    group = w.num_qo_heads // w.num_kv_heads
    lens = request_lengths(w.qo_indptr, w.kv_page_indptr, w.kv_last_page_len, w.page_size)
    qo_indptr = np.asarray(w.qo_indptr, np.int64)
    indices = np.asarray(w.kv_page_indices, np.int64)
    by_group: Dict[Tuple[int, int], List[Tuple[int, int]]] = {}
    for (row, h) in rows:
        b = request_of_row(qo_indptr, row)
        by_group.setdefault((b, kv_head_of(h, group)), []).append((row, h))
    res = {}
    for (b, g), items in by_group.items():
        qo, kv, p0, npg = lens[b]
        K, V = gather_kv(w.kv_cache, indices[p0:p0 + npg], kv, g, w.page_size)
        Qr = np.stack([_as_f64(w.q[row, h]) for (row, h) in items])
        nvis = np.array([visible_keys(kv, qo, row - int(qo_indptr[b]), w.causal) for (row, _) in items])
        o, l = _rows_attention(Qr, K, V, nvis, scale)
        for j, key in enumerate(items):
            res[key] = (o[j], float(l[j]))
    return res


# ---------------------------------------------------------------------------
# split-KV partial states and their merge


def partial_state(Qr: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """(o, lse) of rows ``Qr`` over one slice of keys: o normalised by its own
    softmax sum; a slice with no key gives o = 0 and lse = -inf."""
    if K.shape[0] == 0:
        return np.zeros((Qr.shape[0], V.shape[1])), np.full(Qr.shape[0], -np.inf)
    nvis = np.full(Qr.shape[0], K.shape[0])
    return _rows_attention(Qr, K, V, nvis, scale)


def merge_states(os_: Sequence[np.ndarray], lses: Sequence[np.ndarray]):
    """Combine per-slice states of the same rows: each slice's softmax sum is
    exp(lse_s), so the whole sum is sum_s exp(lse_s) and each slice output is
    weighted by its share of it.  Slices with lse = -inf weigh nothing."""
    L = np.stack([np.asarray(x, np.float64) for x in lses])          # [S, R]
    O = np.stack([np.asarray(x, np.float64) for x in os_])           # [S, R, D]
    M = L.max(axis=0)                                                # [R]
    Mf = np.where(np.isfinite(M), M, 0.0)
    W = np.exp(L - Mf[None, :])                                      # [S, R]
    Z = W.sum(axis=0)
    lse = np.where(Z > 0, Mf + np.log(np.where(Z > 0, Z, 1.0)), -np.inf)
    out = np.einsum("sr,srd->rd", W, O) / np.where(Z > 0, Z, 1.0)[:, None]
    return out, lse


# ---------------------------------------------------------------------------
# the page-table walk itself


def gather_index_table(kv_page_indptr, kv_page_indices, kv_last_page_len, page_size):
    """For every request b and logical token t < kv_b (in request order),
    the physical (page, slot) holding it: two int32 arrays of length sum kv_b."""
    lens = request_lengths(np.zeros(len(kv_page_indptr), np.int64), kv_page_indptr,
                           kv_last_page_len, page_size)
    indices = np.asarray(kv_page_indices, np.int64)
    pages, slots = [], []
    for (_, kv, p0, npg) in lens:
        pl = indices[p0:p0 + npg]
        for t in range(kv):
            p, s = locate(pl, t, page_size)
            pages.append(p)
            slots.append(s)
    return np.array(pages, np.int32), np.array(slots, np.int32)
