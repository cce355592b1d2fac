"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics.

Each check compares the oracle with something other than itself -- a
closed form, a library routine on a special case (torch's
scaled_dot_product_attention on contiguous pages), an invariant of the
definition, brute force, or a value printed on the pages (tests/golden).
``test_planted_mistakes`` then swaps each named helper of the oracle for a
plausible mistake and requires at least one pin to fail.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads
from oracle import attention as A
from oracle import plan_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small(qo, kv, Hq, Hkv, D=16, ps=4, dtype=torch.float16, causal=True, seed=7, extra_pages=3):
    return workloads.make_custom("t", qo, kv, Hq, Hkv, D, ps, dtype=dtype, causal=causal,
                                 seed=seed, extra_pages=extra_pages)


def dense_reference(w):
    """Per request: contiguous K/V built by indexing the cache, then torch's
    scaled_dot_product_attention (fp64) with an explicit bottom-right mask,
    and torch.logsumexp for the lse.  Independent of the oracle's code."""
    T, Hq, D = w.q.shape
    G = w.num_qo_heads // w.num_kv_heads
    out = np.zeros((T, Hq, D))
    lse = np.zeros((T, Hq))
    for b in range(w.batch_size):
        q0, q1 = int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])
        p0, p1 = int(w.kv_page_indptr[b]), int(w.kv_page_indptr[b + 1])
        kv = int(w.gen_kv_lens[b])
        qo = q1 - q0
        if qo == 0:
            continue
        pages = torch.from_numpy(w.kv_page_indices[p0:p1].astype(np.int64))
        blk = w.kv_cache.index_select(0, pages).to(torch.float64)      # [np, 2, ps, Hkv, D]
        K = blk[:, 0].reshape(-1, w.num_kv_heads, D)[:kv]                 # [kv, Hkv, D]
        V = blk[:, 1].reshape(-1, w.num_kv_heads, D)[:kv]
        K = K.repeat_interleave(G, dim=1).transpose(0, 1)                 # [Hq, kv, D]
        V = V.repeat_interleave(G, dim=1).transpose(0, 1)
        Q = w.q[q0:q1].to(torch.float64).transpose(0, 1)                  # [Hq, qo, D]
        i = torch.arange(qo)[:, None]
        j = torch.arange(kv)[None, :]
        mask = (j <= kv - qo + i) if w.causal else torch.ones(qo, kv, dtype=torch.bool)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
        s = (Q @ K.transpose(1, 2)) / math.sqrt(D)
        s = s.masked_fill(~mask, float("-inf"))
        out[q0:q1] = o.transpose(0, 1).numpy()
        lse[q0:q1] = torch.logsumexp(s, dim=-1).transpose(0, 1).numpy()
    return out, lse


def close(a, b, tol=1e-10):
    return np.allclose(a, b, rtol=0, atol=tol)


# ---------------------------------------------------------------------------
# pins, each a function returning True when the oracle agrees


def pin_sdpa_contiguous():
    ok = True
    for causal in (True, False):
        for (Hq, Hkv) in ((2, 1), (4, 2), (6, 3)):
            w = small([1, 3, 6, 0, 9], [7, 5, 6, 2, 13], Hq, Hkv, causal=causal, seed=11 + Hq)
            w2 = workloads.make_custom("c", [1, 3, 6, 0, 9], [7, 5, 6, 2, 13], Hq, Hkv, 16, 4,
                                       causal=causal, seed=11 + Hq, permute_pages=False)
            for ww in (w, w2):
                o, l = A.attention(ww)
                ro, rl = dense_reference(ww)
                rows = np.repeat(ww.qo_lens() > 0, ww.qo_lens())
                ok &= close(o[rows], ro[rows]) and close(l[rows], rl[rows])
    # head_dim 256 (scale 1/16), pages of 4 slots
    w3 = workloads.make_custom("c256", [1, 4, 0, 7], [9, 6, 3, 7], 4, 2, 256, 4, seed=19)
    o, l = A.attention(w3)
    ro, rl = dense_reference(w3)
    rows = np.repeat(w3.qo_lens() > 0, w3.qo_lens())
    ok &= close(o[rows], ro[rows]) and close(l[rows], rl[rows])
    return bool(ok)


def pin_walk_equals_gather():
    w = workloads.tiny()
    o1, l1 = A.attention(w, "walk")
    o2, l2 = A.attention(w, "gather")
    w = small([2, 1, 4], [9, 3, 4], 4, 2, causal=False, seed=3)
    o3, l3 = A.attention(w, "walk")
    o4, l4 = A.attention(w, "gather")
    return close(o1, o2) and close(l1, l2) and close(o3, o4) and close(l3, l4)


def pin_single_key_returns_v():
    # qo == kv, causal: row 0 sees only key 0 -> out = V[0] exactly, lse = scale*q.k
    w = small([5], [5], 2, 1, D=32, ps=2, seed=21)
    o, l = A.attention(w)
    p0 = int(w.kv_page_indices[0])
    ok = True
    for h in range(2):
        v0 = w.kv_cache[p0, 1, 0, 0].double().numpy()
        k0 = w.kv_cache[p0, 0, 0, 0].double().numpy()
        ok &= np.array_equal(o[0, h], v0)
        ok &= abs(l[0, h] - float(np.dot(w.q[0, h].double().numpy(), k0)) / math.sqrt(32)) < 1e-12
    return bool(ok)


def pin_constant_v():
    w = small([3, 1], [9, 6], 4, 2, D=16, ps=4, seed=5)
    c = torch.randn(16, generator=torch.Generator().manual_seed(1)).to(torch.float16)
    w.kv_cache[:, 1] = c
    o, _ = A.attention(w)
    return close(o, np.broadcast_to(c.double().numpy(), o.shape), 1e-12)


def pin_zero_query():
    # q = 0: every visible key weighs the same -> out = mean of visible V, lse = ln n
    w = small([4, 1], [6, 5], 2, 1, D=8, ps=2, seed=9)
    w.q.zero_()
    o, l = A.attention(w)
    ok = True
    for b, (qo, kv) in enumerate([(4, 6), (1, 5)]):
        p0, p1 = int(w.kv_page_indptr[b]), int(w.kv_page_indptr[b + 1])
        V = w.kv_cache[torch.from_numpy(w.kv_page_indices[p0:p1].astype(np.int64)), 1, :, 0]
        V = V.reshape(-1, 8)[:kv].double().numpy()
        for i in range(qo):
            n = kv - qo + i + 1
            row = int(w.qo_indptr[b]) + i
            for h in range(2):
                ok &= close(o[row, h], V[:n].mean(0), 1e-12) and abs(l[row, h] - math.log(n)) < 1e-12
    return bool(ok)


def pin_two_keys_closed_form():
    # one decode row over two keys, values picked by hand
    D = 4
    qv = torch.tensor([[[1.0, 0.0, 2.0, 0.0]]], dtype=torch.float16)
    cache = torch.zeros((1, 2, 2, 1, D), dtype=torch.float16)
    cache[0, 0, 0, 0] = torch.tensor([1.0, 1.0, 1.0, 1.0])
    cache[0, 0, 1, 0] = torch.tensor([0.0, 2.0, -1.0, 4.0])
    cache[0, 1, 0, 0] = torch.tensor([3.0, 0.0, 0.0, 1.0])
    cache[0, 1, 1, 0] = torch.tensor([-1.0, 2.0, 0.5, 0.0])
    o, l = A.attention_gather(qv, cache, [0, 1], [0, 1], [0], [2], 1, 1, D, 2)
    s0, s1 = 3.0 / 2.0, -2.0 / 2.0                       # scale 1/sqrt(4)
    z = math.exp(s0) + math.exp(s1)
    v0, v1 = np.array([3.0, 0, 0, 1]), np.array([-1.0, 2, 0.5, 0])
    want = (math.exp(s0) * v0 + math.exp(s1) * v1) / z
    return close(o[0, 0], want, 1e-12) and abs(l[0, 0] - math.log(z)) < 1e-12


def pin_page_permutation():
    w = small([3, 1, 5], [10, 7, 5], 4, 2, D=16, ps=4, seed=13)
    o, l = A.attention(w)
    perm = workloads.randperm(w.num_pages, 99).astype(np.int64)
    cache2 = torch.empty_like(w.kv_cache)
    cache2[torch.from_numpy(perm)] = w.kv_cache
    w.kv_cache = cache2
    w.kv_page_indices = perm[w.kv_page_indices].astype(np.int32)
    o2, l2 = A.attention(w)
    return np.array_equal(o, o2) and np.array_equal(l, l2)


def pin_prefix_sharing():
    a = workloads.prefix(batch_size=3)
    b = workloads.prefix(duplicated=True, batch_size=3)
    oa, la = A.attention(a)
    ob, lb = A.attention(b)
    return np.array_equal(oa, ob) and np.array_equal(la, lb)


def pin_decode_equals_last_prefill_row():
    # the last row of a causal prefill equals a qo=1 decode of the same request
    w = small([6, 3], [6, 9], 4, 1, D=16, ps=4, seed=17)
    o, l = A.attention(w)
    ok = True
    for b in range(2):
        last = int(w.qo_indptr[b + 1]) - 1
        q1 = w.q[last:last + 1].clone()
        od, ld = A.attention_gather(q1, w.kv_cache, [0, 1], w.kv_page_indptr[b:b + 2] - w.kv_page_indptr[b],
                                    w.kv_page_indices[w.kv_page_indptr[b]:w.kv_page_indptr[b + 1]],
                                    w.kv_last_page_len[b:b + 1], 4, 1, 16, 4)
        ok &= close(od[0], o[last], 1e-12) and close(ld[0], l[last], 1e-12)
    return bool(ok)


def pin_padded_equals_unpadded():
    a = workloads.ragged(batch_size=4)
    b = workloads.ragged(padded=True, batch_size=4)
    oa, la = A.attention(a)
    ob, lb = A.attention(b)
    ok = True
    for r in range(4):
        L = int(a.qo_indptr[r + 1] - a.qo_indptr[r])
        ra = slice(int(a.qo_indptr[r]), int(a.qo_indptr[r + 1]))
        rb = slice(200 * r, 200 * r + L)
        # equal up to fp64 rounding: BLAS may block a 200-key product differently
        ok &= close(oa[ra], ob[rb], 1e-12) and close(la[ra], lb[rb], 1e-12)
    return bool(ok)


def pin_split_merge():
    w = small([1, 4], [19, 12], 4, 2, D=16, ps=4, seed=23)
    o, l = A.attention(w)
    scale = 1 / math.sqrt(16)
    ok = True
    for b in range(2):
        qo, kv = int(w.qo_lens()[b]), int(w.gen_kv_lens[b])
        p0, p1 = int(w.kv_page_indptr[b]), int(w.kv_page_indptr[b + 1])
        for g in range(2):
            K, V = A.gather_kv(w.kv_cache, w.kv_page_indices[p0:p1], kv, g, 4)
            for h in (2 * g, 2 * g + 1):
                for i in range(qo):
                    row = int(w.qo_indptr[b]) + i
                    n = kv - qo + i + 1
                    Qr = w.q[row:row + 1, h].double().numpy()
                    cuts = [0, 4, 8, n] if n > 8 else [0, 4, n]
                    parts = [A.partial_state(Qr, K[c0:c1], V[c0:c1], scale) for c0, c1 in zip(cuts[:-1], cuts[1:])]
                    parts.append(A.partial_state(Qr, K[:0], V[:0], scale))     # an empty split
                    mo, ml = A.merge_states([p[0] for p in parts], [p[1] for p in parts])
                    ok &= close(mo[0], o[row, h], 1e-12) and abs(ml[0] - l[row, h]) < 1e-12
                    # two-way merge: lse is log(exp(lse1) + exp(lse2))
                    l1 = parts[0][1][0]
                    l2 = A.merge_states([parts[1][0]], [parts[1][1]])[1][0] if len(parts) > 2 else -np.inf
                    ok &= abs(A.merge_states([parts[0][0], parts[1][0]], [parts[0][1], parts[1][1]])[1][0]
                              - np.logaddexp(l1, l2)) < 1e-12
    return bool(ok)


def pin_kv_len_matches_generator():
    ok = True
    for w in (workloads.tiny(), workloads.decode(batch_size=4), workloads.ragged(batch_size=6),
              workloads.prefix(batch_size=2)):
        lens = A.request_lengths(w.qo_indptr, w.kv_page_indptr, w.kv_last_page_len, w.page_size)
        ok &= [kv for (_, kv, _, _) in lens] == [int(x) for x in w.gen_kv_lens]
    return bool(ok)


def pin_gather_walk_golden():
    # (page, slot) of every token of the tiny batch, brute force from the tables
    w = workloads.tiny()
    pages, slots = A.gather_index_table(w.kv_page_indptr, w.kv_page_indices, w.kv_last_page_len, 4)
    ok = len(pages) == 8 + 13 + 17 + 24
    k = 0
    for b, kv in enumerate([8, 13, 17, 24]):
        p0 = int(w.kv_page_indptr[b])
        for t in range(kv):
            ok &= pages[k] == w.kv_page_indices[p0 + t // 4] and slots[k] == t % 4
            k += 1
    return bool(ok)


def pin_sampled_rows():
    """attention_rows (the sampled-row form the full-size checks use) against
    torch's scaled_dot_product_attention on contiguous K/V and against the
    whole-batch oracle, element by element.  The batch puts empty requests
    (qo_len 0) between non-empty ones and ends on a one-row request, so rows
    at every request boundary are mapped to their request; G = 2, causal
    and not, pages permuted; rows are asked for out of order."""
    ok = True
    for causal in (True, False):
        w = small([2, 0, 3, 0, 0, 1, 4, 1], [5, 4, 7, 3, 1, 9, 6, 2], 4, 2, causal=causal, seed=23)
        T = int(w.qo_indptr[-1])
        rows = [(r, h) for r in range(T) for h in range(w.num_qo_heads)]
        order = np.random.default_rng(5).permutation(len(rows))
        rows = [rows[i] for i in order]
        got = A.attention_rows(w, rows)
        ro, rl = dense_reference(w)
        fo, fl = A.attention(w)
        for (r, h) in rows:
            o, l = got[(r, h)]
            ok &= close(o, ro[r, h], 1e-12) and abs(l - rl[r, h]) <= 1e-12
            ok &= close(o, fo[r, h], 1e-12) and abs(l - fl[r, h]) <= 1e-12
    return bool(ok)


PINS = [pin_sdpa_contiguous, pin_walk_equals_gather, pin_single_key_returns_v, pin_constant_v,
        pin_zero_query, pin_two_keys_closed_form, pin_page_permutation, pin_prefix_sharing,
        pin_decode_equals_last_prefill_row, pin_padded_equals_unpadded, pin_split_merge,
        pin_kv_len_matches_generator, pin_gather_walk_golden, pin_sampled_rows]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin()


# ---------------------------------------------------------------------------
# the pages' own numbers: the decode timing script


def test_golden_decode_script():
    g = json.load(open(os.path.join(GOLDEN, "decode_script.json")))
    p = g["params"]
    ps, seq, B = p["page_size"], p["seq_length"], p["batch_size"]
    pages_per_seq = (seq + ps - 1) // ps
    assert pages_per_seq == g["expect"]["num_pages_per_seq"]
    assert pages_per_seq * B == g["expect"]["max_num_pages"]
    assert p["num_qo_heads"] // p["num_kv_heads"] == g["expect"]["group_size"]
    indptr = np.arange(0, pages_per_seq * B + 1, pages_per_seq)
    # the script's literal last_page_len (seq % page_size = 0) breaks its own
    # 1 <= last <= page_size rule: rejected
    with pytest.raises(A.PlanError):
        A.request_lengths(np.arange(B + 1), indptr, np.full(B, seq % ps), ps)
    # a full last page gives back seq_length keys per request
    lens = A.request_lengths(np.arange(B + 1), indptr, np.full(B, ps), ps)
    assert all(kv == g["expect"]["kv_len"] for (_, kv, _, _) in lens)
    w = workloads.decode()
    assert w.kv_cache.shape == tuple(g["expect"]["kv_cache_shape"])


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail


MUTANTS = {
    "gqa_interleaved": ("kv_head_of", lambda h, group: h % 2),
    "mask_top_left": ("visible_keys", lambda kv, qo, i, causal: (i + 1) if causal else kv),
    "mask_off_by_one": ("visible_keys", lambda kv, qo, i, causal: (kv - qo + i) if causal else kv),
    "scale_1_over_d": ("default_scale", lambda D: 1.0 / D),
    "slot_swapped": ("locate", lambda pages, t, ps: (int(pages[t % len(pages)]), t // len(pages) % ps)),
    "kv_len_ignores_last": ("kv_len_of", lambda n, last, ps: n * ps),
    "lse_base2": ("softmax_stats", lambda s: (lambda m: (m + math.log2(np.sum(np.exp(s - m))), np.exp(s - m) / np.sum(np.exp(s - m))))(float(np.max(s)))),
    # sampled rows: a row at a request boundary given to the request before it
    "row_request_left": ("request_of_row",
                         lambda qo_indptr, row: int(np.searchsorted(np.asarray(qo_indptr), row, side="left") - 1)),
    # sampled rows: the first request's row index used for every request
    "row_request_first": ("request_of_row", lambda qo_indptr, row: 0),
    "no_max_shift_weights": ("softmax_stats", lambda s: (float(np.max(s)) + math.log(np.sum(np.exp(s - np.max(s)))), np.exp(s - np.max(s)))),
}


@pytest.mark.parametrize("name", sorted(MUTANTS) + ["kv_swapped"])
def test_planted_mistakes(name, monkeypatch):
    if name == "kv_swapped":
        monkeypatch.setattr(A, "K_SLOT", 1)
        monkeypatch.setattr(A, "V_SLOT", 0)
    else:
        attr, fn = MUTANTS[name]
        monkeypatch.setattr(A, attr, fn)
    failed = []
    for pin in PINS:
        try:
            if not pin():
                failed.append(pin.__name__)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"


# ---------------------------------------------------------------------------
# plan restatement: brute-force coverage of every (row, head, key) once


@pytest.mark.parametrize("wname,sms,kw", [
    ("tiny", 148, {}), ("tiny", 2, {"prefill_chunk_tiles": 1}), ("decode", 148, {}),
    ("ragged", 148, {}), ("prefix", 148, {}), ("tiny", 148, {"force_prefill": True}),
    ("custom_long", 4, {}), ("smallq", 4, {}), ("smallq", 148, {"decode_cuda_cores": True}),
    ("smallq_g16", 148, {}), ("smallq_g1", 3, {}), ("d256", 148, {}), ("d256", 3, {"decode_chunk_pages": 2}),
    ("ragged", 148, {"prefill_q_tiles": 1}), ("custom_long", 4, {"prefill_q_tiles": 1}),
    ("custom_long", 4, {"prefill_q_tiles": 2}),
])
def test_plan_ref_covers_every_pair_once(wname, sms, kw):
    if wname == "d256":  # G 4 at head_dim 256: one-token decodes, a 5-token request, 1- and 3-tile prefills
        w = small([1, 70, 1, 5, 100], [1, 70, 300, 200, 400], 8, 2, D=256, ps=8, seed=7)
    elif wname == "custom_long":
        w = small([1, 40, 1, 300], [2000, 700, 33, 300], 8, 2, D=64, ps=16, seed=3)
    elif wname == "smallq":  # G 8: rows 32, 32, 16, 8, 64, and a prefill of 9 tokens
        w = small([4, 4, 2, 1, 8, 9], [300, 40, 900, 70, 500, 9], 16, 2, D=64, ps=16, seed=4)
    elif wname == "smallq_g16":  # G 16: rows 16, 32, 64, then prefill
        w = small([1, 2, 4, 5], [77, 500, 260, 30], 16, 1, D=64, ps=8, seed=5)
    elif wname == "smallq_g1":  # G 1: up to 64 tokens per small-query item
        w = small([64, 65, 3, 1], [64, 200, 1000, 9], 2, 2, D=64, ps=4, seed=6)
    elif wname == "decode":
        w = workloads.decode(batch_size=16)
    elif wname == "ragged":
        w = workloads.ragged(batch_size=8)
    elif wname == "prefix":
        w = workloads.prefix(batch_size=4)
    else:
        w = workloads.tiny()
    blob = plan_ref.build(**{k: v for k, v in w.plan_args().items() if k != "causal"}, causal=w.causal,
                          dtype=plan_ref.FP16 if w.dtype == torch.float16 else plan_ref.BF16,
                          num_sms=sms, **kw)
    h = plan_ref.decode_header(blob)
    dec, pre, mer = plan_ref.items(blob)
    G = h["G"]
    Hq = h["Hq"]
    cover = {}
    lens = A.request_lengths(w.qo_indptr, w.kv_page_indptr, w.kv_last_page_len, w.page_size)
    for (b, hk, t0, t1, pr, *_r) in dec:
        qo, kv = lens[b][0], lens[b][1]
        assert qo * G <= 32
        for i in range(qo):
            vis = kv - qo + i + 1 if w.causal else kv
            row = int(w.qo_indptr[b]) + i
            for g in range(G):
                for t in range(t0, min(t1, vis)):
                    key = (row, hk * G + g, t)
                    assert key not in cover
                    cover[key] = 1
    for (b, hk, qt0, n, k0, k1, pr, _) in pre:
        qo, kv = lens[b][0], lens[b][1]
        for i in range(qt0, qt0 + n):
            vis = kv - qo + i + 1 if w.causal else kv
            row = int(w.qo_indptr[b]) + i
            for g in range(G):
                for t in range(k0, min(k1, vis)):
                    key = (row, hk * G + g, t)
                    assert key not in cover
                    cover[key] = 1
    want = 0
    for b, (qo, kv, _, _) in enumerate(lens):
        for i in range(qo):
            want += (kv - qo + i + 1 if w.causal else kv) * Hq
    assert len(cover) == want
    # partial rows are distinct and every merge entry points inside the pool
    rows = set()
    for (o0, p0, ns, st) in mer:
        for s in range(ns):
            for g in range(G):
                r = p0 + s * st + g
                assert 0 <= r < h["n_part_rows"] and r not in rows
                rows.add(r)
    assert len(rows) == h["n_part_rows"]
    # decode items: grouped by row class (counts in the header), longest first within a class
    cls = np.array([next(c for c, n in enumerate((8, 16, 32, 64)) if lens[b][0] * G <= n) for b in dec[:, 0]],
                   np.int64)
    assert all(np.diff(cls) >= 0)
    assert h["dec_class_items"] == [int((cls == c).sum()) for c in range(4)]
    for c in range(4):
        ln = (dec[:, 3] - dec[:, 2])[cls == c]
        assert all(np.diff(ln) <= 0)
    assert all(np.diff(pre[:, 5] - pre[:, 4]) <= 0) if len(pre) else True


def test_plan_ref_decode_script_split():
    w = workloads.decode()
    blob = plan_ref.build(**{k: v for k, v in w.plan_args().items() if k != "causal"},
                          dtype=plan_ref.FP16, num_sms=148)
    h = plan_ref.decode_header(blob)
    # at the largest chunk (2048 keys = 128 pages) every request is one item: 128 items fit one
    # wave of 2 * 148 and cover more than 3/4 of the 148 SMs, so no request is split
    assert h["dec_chunk_pages"] == 128 and h["n_dec"] == 128 and h["n_merge"] == 0
    assert h["n_part_rows"] == 0 and h["n_pre"] == 0
    dec, _, _ = plan_ref.items(blob)
    assert sorted({(int(a), int(b)) for a, b in dec[:, 2:4]}) == [(0, 1024)]
    # on 256 SMs the 128 items would leave half of them idle: split in two (one wave of 512)
    blob = plan_ref.build(**{k: v for k, v in w.plan_args().items() if k != "causal"},
                          dtype=plan_ref.FP16, num_sms=256)
    h = plan_ref.decode_header(blob)
    assert h["dec_chunk_pages"] == 16 and h["n_dec"] == 512 and h["n_merge"] == 128


@pytest.mark.parametrize("kw", [{}, {"prefill_chunk_tiles": 1, "decode_chunk_pages": 2}])
def test_plan_ref_cascade_covers_every_pair_once(kw):
    """Shared-prefix cascade plans: every (query token, head, key) of the
    flattened sequence (prefix pages, then the request's own) is covered by
    exactly one item -- the group's prefix items for prefix keys, the
    request's items for its own -- and every partial row an item writes is
    read by exactly one merge entry of its token."""
    w = workloads.make_custom("t", [3, 1, 20, 2, 1], [40, 70, 60, 300, 30], 8, 2, 64, 4, seed=9,
                              permute_pages=False)
    ind, ptr = w.kv_page_indices.copy(), w.kv_page_indptr
    for b in (1, 2):                      # requests 0-2 share 5 pages, requests 3-4 share 2
        ind[ptr[b]:ptr[b] + 5] = ind[ptr[0]:ptr[0] + 5]
    ind[ptr[4]:ptr[4] + 2] = ind[ptr[3]:ptr[3] + 2]
    w.kv_page_indices = ind
    gind, npre = [0, 3, 5], [5, 2]
    groups, args = workloads.split_prefix(w, gind, npre)
    blob = plan_ref.build(**{k: v for k, v in args.items() if k != "causal"}, causal=w.causal,
                          dtype=plan_ref.FP16, num_sms=3, prefix_groups=groups, **kw)
    h = plan_ref.decode_header(blob)
    dec, pre, mer = plan_ref.items(blob)
    G, Hq, ps, B = h["G"], h["Hq"], w.page_size, w.batch_size
    own = A.request_lengths(args["qo_indptr"], args["kv_page_indptr"], args["kv_last_page_len"], ps)
    pre_len = {b: npre[g] * ps for g in range(2) for b in range(gind[g], gind[g + 1])}
    qi = np.asarray(w.qo_indptr)
    tok_req = {int(qi[b]) + i: (b, i) for b in range(B) for i in range(own[b][0])}
    cover, writes = {}, {}

    def add(tok, head, key):
        k = (tok, head, key)
        assert k not in cover
        cover[k] = 1

    for (b, hk, t0, t1, pr, *_r) in dec:
        qo, kv = own[b][0], own[b][1]
        for i in range(qo):
            for g in range(G):
                for t in range(t0, min(t1, kv - qo + i + 1)):
                    add(int(qi[b]) + i, hk * G + g, pre_len[b] + t)
                if pr >= 0:
                    writes[pr + i * G + g] = (int(qi[b]) + i, hk * G + g)
    for (b, hk, q0, n, k0, k1, pr, _) in pre:
        for i in range(q0, q0 + n):
            for g in range(G):
                if b >= B:                       # a group's prefix: every prefix key visible
                    r0 = gind[b - B]
                    tok = int(qi[r0]) + i
                    keys = range(k0, k1)
                else:
                    qo, kv = own[b][0], own[b][1]
                    tok = int(qi[b]) + i
                    keys = [pre_len[b] + t for t in range(k0, min(k1, kv - qo + i + 1))]
                for key in keys:
                    add(tok, hk * G + g, key)
                if pr >= 0:
                    writes[pr + (i - q0) * G + g] = (tok, hk * G + g)
    want = sum((pre_len[b] + own[b][1] - own[b][0] + i + 1) * Hq for b in range(B) for i in range(own[b][0]))
    assert len(cover) == want
    read = {}
    for (o0, p0, ns, st) in mer:
        tok, hk = divmod(o0, Hq)
        for s in range(ns):
            for g in range(G):
                r = p0 + s * st + g
                assert r not in read
                read[r] = (tok, hk + g)
    assert all(read.get(r) == th for r, th in writes.items())   # every written row merged into its own token
