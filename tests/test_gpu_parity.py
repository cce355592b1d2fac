"""GPU parity: the CUDA path, called through the C ABI, against the fp64
oracle on the same seeded inputs, plus the invariants that must hold
bit-exactly on the GPU (page placement, prefix sharing) and edge cases."""
import dataclasses

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A
from oracle import plan_ref

pytestmark = pytest.mark.gpu

pa = pytest.importorskip("attention_paged_kv_gb300")
from parity import assert_close, run  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    pa.load()


# ---------------------------------------------------------------- workloads


@pytest.mark.parametrize("opts", [{}, {"force_prefill": True}, {"decode_chunk_pages": 1},
                                  {"prefill_chunk_tiles": 1, "decode_chunk_pages": 1}])
def test_tiny_all_paths(opts):
    w = workloads.tiny()
    ro, rl = A.attention(w, "walk")
    out, lse, _ = run(w, **opts)
    assert_close(out, lse, ro, rl, w.dtype, what=f"tiny {opts}")


@pytest.mark.parametrize("opts", [{}, {"decode_chunk_pages": 64}, {"decode_chunk_pages": 1},
                                  {"decode_cuda_cores": True}, {"decode_cuda_cores": True, "decode_chunk_pages": 1}])
def test_decode_script_batch(opts):
    w = workloads.decode()
    ro, rl = A.attention(w)
    out, lse, plan = run(w, **opts)
    assert_close(out, lse, ro, rl, w.dtype, what=f"decode {opts}")


@pytest.mark.parametrize("cuda_cores", [False, True])
def test_decode_equals_prefill_qo1(cuda_cores):
    """The timing script's closing check: decode output allclose to the
    prefill kernel's output on the same qo_len = 1 batch (atol = rtol = 1e-3)."""
    w = workloads.decode()
    o_dec, l_dec, _ = run(w, decode_cuda_cores=cuda_cores)
    o_pre, l_pre, _ = run(w, force_prefill=True)
    assert np.allclose(o_dec, o_pre, atol=1e-3, rtol=1e-3)
    assert np.allclose(l_dec, l_pre, atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("opts", [{}, {"decode_cuda_cores": True}, {"force_prefill": True},
                                  {"force_cp_async": True, "force_prefill": True}])
@pytest.mark.parametrize("ps", [4, 16, 128])
def test_nan_outside_the_kv_range(opts, ps):
    """Slots past each request's last_page_len and pages no request uses
    hold NaN: no kernel may let them reach an output (masked keys still
    meet V in the P V product, where 0 * NaN would be NaN)."""
    lens = [1, 63, 64, 65, 127, 129, 200, 1000, 100, 300, 129, 300, 500]
    qo = [1] * 8 + [40, 130] + [2, 4, 8]  # the last three: 2, 4, 8 tokens x 8 heads, small-query items
    w = workloads.make_custom("nan", qo, lens, 16, 2, 128, ps, dtype=torch.bfloat16, seed=ps + 3, extra_pages=5)
    used = torch.zeros(w.num_pages, dtype=torch.bool)
    kv = w.kv_cache.clone()
    for b in range(len(lens)):
        pages = torch.as_tensor(np.asarray(w.kv_page_indices[w.kv_page_indptr[b]:w.kv_page_indptr[b + 1]]),
                                dtype=torch.long)
        used[pages] = True
        kv[int(pages[-1]), :, int(w.kv_last_page_len[b]):] = float("nan")
    kv[~used] = float("nan")
    w = dataclasses.replace(w, kv_cache=kv)
    ro, rl = A.attention(w)
    assert np.isfinite(ro).all()
    out, lse, _ = run(w, **opts)
    assert_close(out, lse, ro, rl, w.dtype, what=f"NaN outside range {opts} ps {ps}")


def test_ragged_prefill():
    w = workloads.ragged()
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, w.dtype, what="ragged")


def test_ragged_padded_equals_unpadded():
    a = workloads.ragged()
    b = workloads.ragged(padded=True)
    oa, la, _ = run(a)
    ob, lb, _ = run(b)
    ro, rl = A.attention(a)
    for r in range(a.batch_size):
        L = int(a.qo_indptr[r + 1] - a.qo_indptr[r])
        ra = slice(int(a.qo_indptr[r]), int(a.qo_indptr[r + 1]))
        rb = slice(200 * r, 200 * r + L)
        assert_close(ob[rb], lb[rb], ro[ra], rl[ra], a.dtype, what=f"padded request {r}")
        assert np.allclose(oa[ra], ob[rb], atol=1e-2, rtol=0)


def test_ragged_cp_async_equals_tma():
    w = workloads.ragged()
    o1, l1, _ = run(w)
    o2, l2, _ = run(w, force_cp_async=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_prefix_shared():
    w = workloads.prefix()
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, w.dtype, what="prefix")


def test_prefix_shared_equals_duplicated_bitexact():
    a, b = workloads.prefix(), workloads.prefix(duplicated=True)
    oa, la, _ = run(a)
    ob, lb, _ = run(b)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


@pytest.mark.parametrize("name", ["ragged", "mixed_small", "tiny"])
def test_page_permutation_bitexact(name):
    w = workloads.ragged() if name == "ragged" else (
        workloads.tiny() if name == "tiny" else workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000))
    o1, l1, _ = run(w)
    perm = workloads.randperm(w.num_pages, 4242).astype(np.int64)
    cache2 = torch.empty_like(w.kv_cache)
    cache2[torch.from_numpy(perm)] = w.kv_cache
    w.kv_cache = cache2
    w.kv_page_indices = perm[w.kv_page_indices].astype(np.int32)
    o2, l2, _ = run(w)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_prefill_split_kv():
    w = workloads.make_custom("long", [40, 1, 130, 3], [3000, 1500, 2200, 900], 16, 2, 128, 16,
                              dtype=torch.bfloat16, seed=31)
    ro, rl = A.attention(w)
    o1, l1, p1 = run(w, force_prefill=True)
    o2, l2, p2 = run(w, force_prefill=True, prefill_chunk_tiles=2)
    h = plan_ref.decode_header(p2.dump())
    assert h["n_merge"] > 0
    assert_close(o1, l1, ro, rl, w.dtype, what="unsplit")
    assert_close(o2, l2, ro, rl, w.dtype, what="split")


def test_mixed_step_sampled():
    """The full mixed batch (8192-token prefill + 256 decodes) on the GPU,
    checked on sampled rows the oracle computes one by one."""
    w = workloads.mixed()
    out, lse, _ = run(w)
    Hq = w.num_qo_heads
    pre_tokens = [0, 1, 15, 16, 17, 127, 128, 129, 1000, 2047, 4095, 4096, 6001, 8190, 8191]
    rows = [(t, h) for t in pre_tokens for h in range(Hq)]
    dec_reqs = [1, 2, 3, 50, 100, 200, 255, 256]
    rows += [(int(w.qo_indptr[b]), h) for b in dec_reqs for h in range(Hq)]
    ref = A.attention_rows(w, rows)
    ro = np.stack([ref[k][0] for k in rows])
    rl = np.array([ref[k][1] for k in rows])
    go = np.stack([out[r, h] for (r, h) in rows])
    gl = np.array([lse[r, h] for (r, h) in rows])
    assert_close(go, gl, ro, rl, w.dtype, what="mixed sampled")
    assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---------------------------------------------------------------- indexing / metadata


@pytest.mark.parametrize("name", ["tiny", "ragged", "mixed_small"])
def test_gather_indices_bitexact(name):
    w = workloads.ragged() if name == "ragged" else (
        workloads.tiny() if name == "tiny" else workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000))
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype)
    pages, slots = plan.debug_gather()
    torch.cuda.synchronize()
    rp, rs = A.gather_index_table(w.kv_page_indptr, w.kv_page_indices, w.kv_last_page_len, w.page_size)
    assert np.array_equal(pages.cpu().numpy(), rp) and np.array_equal(slots.cpu().numpy(), rs)


def test_device_metadata_equals_restated_plan():
    w = workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype)
    want = plan_ref.build(**w.plan_args(), dtype=plan_ref.BF16, num_sms=sms)
    torch.cuda.synchronize()
    dev = plan.workspace[: want.size * 4].cpu().numpy().view(np.int32)
    assert np.array_equal(dev, want)
    assert np.array_equal(plan.dump(), want)


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_shapes_groups_dtypes(dtype, D, G):
    Hkv = 2
    w = workloads.make_custom("s", [1, 7, 1, 33, 0, 140, 1], [1, 7, 300, 200, 5, 333, 64], G * Hkv, Hkv, D, 16,
                              dtype=dtype, seed=G * 100 + D)
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, dtype, what=f"D{D} G{G} {dtype}")
    if G in (4, 8):  # the same batch on the CUDA-core decode kernel
        out, lse, _ = run(w, decode_cuda_cores=True)
        assert_close(out, lse, ro, rl, dtype, what=f"D{D} G{G} {dtype} CUDA-core decode")


SMALLQ = [(1, [32, 2, 9, 1, 17]), (2, [1, 4, 8, 16, 5]), (4, [2, 3, 4, 8, 5]), (8, [1, 2, 3, 4, 2]),
          (16, [1, 2, 1, 2, 2])]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("G,qos", SMALLQ, ids=[f"G{g}" for g, _ in SMALLQ])
@pytest.mark.parametrize("opts", [{}, {"decode_chunk_pages": 2}], ids=["whole", "split"])
def test_small_query(dtype, G, qos, opts):
    """Requests of a few query tokens (qo_len * G <= 32 packed rows, more
    than 128 keys when qo_len > 1) on the warp-MMA kernel: every row class,
    one-token requests from a single key up, each row with its own causal
    limit."""
    extra = [129, 135, 200, 300, 700]
    kvs = [(1 if q == 1 and i == 0 else q + e) for i, (q, e) in enumerate(zip(qos, extra))]
    w = workloads.make_custom("sq", qos, kvs, G * 2, 2, 128, 16, dtype=dtype, seed=G * 7 + len(opts))
    ro, rl = A.attention(w)
    out, lse, plan = run(w, **opts)
    h = plan_ref.decode_header(plan.dump())
    assert h["n_pre"] == 0 and h["dec_cuda_cores"] == 0
    assert_close(out, lse, ro, rl, dtype, what=f"small query G{G} {opts}")


@pytest.mark.parametrize("D,ps,causal", [(64, 4, True), (128, 64, True), (64, 16, False), (128, 1, True)])
def test_small_query_layouts(D, ps, causal):
    """Small-query items at head_dim 64, TMA page rows (64) and cp.async
    pages (1, 4 slots), and without the causal mask."""
    qos, kvs = [4, 3, 1, 2], [200, 170, 300, 1200]
    w = workloads.make_custom("sql", qos, kvs, 16, 2, D, ps, dtype=torch.bfloat16, causal=causal, seed=D + ps)
    ro, rl = A.attention(w)
    for opts in ({}, {"decode_chunk_pages": max(1, 128 // ps)}):
        out, lse, plan = run(w, **opts)
        assert plan_ref.decode_header(plan.dump())["n_pre"] == 0
        assert_close(out, lse, ro, rl, w.dtype, what=f"small query D{D} ps{ps} causal {causal} {opts}")


def test_small_query_equals_prefill_kernel():
    """The speculative-decoding shape on both kernels (atol = rtol = 1e-3 in
    fp16), the small-query analogue of the timing script's closing check."""
    w = workloads.make_custom("sqp", [4] * 12, [40 * i + 130 for i in range(12)], 32, 4, 128, 16, seed=9)
    o1, l1, p1 = run(w)
    o2, l2, p2 = run(w, force_prefill=True)
    assert plan_ref.decode_header(p1.dump())["n_pre"] == 0 and plan_ref.decode_header(p2.dump())["n_dec"] == 0
    assert np.allclose(o1, o2, atol=1e-3, rtol=1e-3)
    assert np.allclose(l1, l2, atol=1e-3, rtol=1e-3)


@pytest.mark.parametrize("ps", [1, 2, 8, 32, 64, 128])
def test_page_sizes(ps):
    w = workloads.make_custom("p", [1, 9, 1, 70], [77, 9, 1, 270], 8, 2, 128, ps, dtype=torch.bfloat16, seed=ps)
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, w.dtype, what=f"page_size {ps}")


def test_non_causal():
    w = workloads.make_custom("nc", [3, 1, 150, 20], [2, 7, 40, 300], 8, 4, 64, 8, causal=False,
                              dtype=torch.float16, seed=77)
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, w.dtype, what="non-causal")


def test_empty_batch_and_empty_requests():
    w = workloads.make_custom("e", [], [], 4, 1, 64, 16, seed=7)
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype)
    out, lse = plan.run(w.q.cuda(), w.kv_cache.cuda())
    torch.cuda.synchronize()
    assert out.numel() == 0
    w = workloads.make_custom("z", [0, 2, 0, 1], [5, 3, 17, 4], 4, 2, 128, 4, seed=8)
    ro, rl = A.attention(w)
    out, lse, _ = run(w)
    assert_close(out, lse, ro, rl, w.dtype, what="empty requests")


def test_single_key_and_constant_v():
    # row 0 of a qo == kv causal request sees one key: out = V[0] exactly
    w = workloads.make_custom("k1", [130, 1], [130, 1], 8, 2, 128, 16, dtype=torch.bfloat16, seed=3)
    out, lse, _ = run(w)
    for b, r in ((0, 0), (1, 130)):
        p0 = int(w.kv_page_indices[w.kv_page_indptr[b]])
        for h in range(8):
            v0 = w.kv_cache[p0, 1, 0, h // 4].double().numpy()
            assert np.array_equal(out[r, h], v0)
    c = torch.randn(128, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    w.kv_cache[:, 1] = c
    out, lse, _ = run(w)
    assert np.allclose(out, np.broadcast_to(c.double().numpy(), out.shape), atol=1e-2, rtol=0)


def test_many_splits_merge():
    """A 32-row small-query request cut into 400 splits (page_size 1, so the
    cp.async path), merged by the merge kernel."""
    w = workloads.make_custom("many", [4], [6400], 16, 2, 128, 1, dtype=torch.bfloat16, seed=22)
    ro, rl = A.attention(w)
    out, lse, plan = run(w, decode_chunk_pages=16)
    h = plan_ref.decode_header(plan.dump())
    assert h["n_dec"] == 2 * 400 and h["dec_class_items"] == [0, 0, 800, 0]
    assert_close(out, lse, ro, rl, w.dtype, what="400 splits")


ONE_TILE = ["tiny", "ragged", "mixed_small", "prefix", "d64_ps1"]


@pytest.mark.parametrize("name", ONE_TILE)
def test_one_tile_prefill_items(name):
    """prefill_q_tiles = 1: prefill items of one 128-row tile, two CTAs to an
    SM (TMA and cp.async pages, head_dim 64 and 128, split-KV)."""
    if name == "tiny":
        w = workloads.tiny()
    elif name == "ragged":
        w = workloads.ragged()
    elif name == "mixed_small":
        w = workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    elif name == "prefix":
        w = workloads.prefix()
    else:
        w = workloads.make_custom("o64", [1, 90, 300, 7], [40, 90, 800, 200], 8, 2, 64, 1, dtype=torch.bfloat16,
                                  seed=41)
    ro, rl = A.attention(w)
    for opts in ({"prefill_q_tiles": 1}, {"prefill_q_tiles": 1, "prefill_chunk_tiles": 1, "force_prefill": True}):
        out, lse, plan = run(w, **opts)
        assert plan_ref.decode_header(plan.dump())["pre_tiles"] == 1
        assert_close(out, lse, ro, rl, w.dtype, what=f"one tile {name} {opts}")


D256_CASES = [(16, {}), (1, {}), (16, {"prefill_chunk_tiles": 1, "decode_chunk_pages": 2}),
              (64, {"force_prefill": True}), (4, {"decode_chunk_pages": 1})]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("ps,opts", D256_CASES, ids=[f"ps{p}-{'-'.join(map(str, o))}" for p, o in D256_CASES])
def test_head_dim_256(dtype, ps, opts):
    """head_dim 256: prefill items of one 128-row tile over several key tiles
    with a ragged tail (and a request whose rows see fewer than 128 keys),
    single-token decode on the CUDA-core kernel, a multi-token small request
    on the prefill kernel, split-KV with the merge, TMA and cp.async pages."""
    qos, kvs = [1, 300, 1, 5, 130, 0, 40], [1, 300, 700, 400, 900, 17, 60]
    w = workloads.make_custom("d256", qos, kvs, 8, 2, 256, ps, dtype=dtype, seed=256 + ps + len(opts))
    ro, rl = A.attention(w)
    out, lse, plan = run(w, **opts)
    h = plan_ref.decode_header(plan.dump())
    if not opts.get("force_prefill"):
        assert h["dec_cuda_cores"] == 1 and h["n_dec"] > 0 and h["n_pre"] > 0
    assert_close(out, lse, ro, rl, dtype, what=f"D256 ps{ps} {opts}")


def _hnd(kv):
    """The same logical cache in the HND layout [P, 2, Hkv, page_size, D]."""
    return kv.permute(0, 1, 3, 2, 4).contiguous()


HND_CASES = [("tiny", {}), ("tiny", {"force_prefill": True}), ("mixed", {}),
             ("mixed", {"decode_chunk_pages": 1, "prefill_chunk_tiles": 1}), ("decode", {"decode_cuda_cores": True}),
             ("smallq", {}), ("ps1", {}), ("ps128", {}), ("mixed", {"force_cp_async": True}), ("d256", {}),
             ("d256", {"force_cp_async": True})]


@pytest.mark.parametrize("name,opts", HND_CASES, ids=[f"{n}-{'-'.join(map(str, o))}" for n, o in HND_CASES])
def test_hnd_layout_equals_nhd_bitexact(name, opts):
    """The HND cache layout reads the same keys and values through other
    addresses: every kernel path gives bit-identical results to NHD."""
    if name == "tiny":
        w = workloads.tiny()
    elif name == "mixed":
        w = workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    elif name == "decode":
        w = workloads.decode(batch_size=16)
    elif name == "smallq":
        w = workloads.make_custom("hq", [4, 2, 8, 1], [300, 700, 200, 90], 16, 2, 128, 16, dtype=torch.bfloat16,
                                  seed=31)
    elif name == "d256":
        w = workloads.make_custom("h256", [1, 140, 1, 3], [500, 300, 90, 200], 16, 2, 256, 16,
                                  dtype=torch.bfloat16, seed=33)
    else:
        ps = int(name[2:])
        w = workloads.make_custom("hp", [1, 9, 1, 70], [77, 9, 300, 270], 8, 2, 128, ps, dtype=torch.bfloat16,
                                  seed=ps + 40)
    o1, l1, _ = run(w, **opts)
    o2, l2, _ = run(w, kv=_hnd(w.kv_cache), kv_layout="HND", **opts)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    if name in ("tiny", "smallq", "d256"):
        ro, rl = A.attention(w)
        assert_close(o2, l2, ro, rl, w.dtype, what=f"HND {name}")


def _cascade_run(w, groups, args, kv=None, **opts):
    plan = pa.Plan(**args, dtype=w.dtype, prefix_groups=groups, **opts)
    out, lse = plan.run(w.q.cuda(), (w.kv_cache if kv is None else kv).cuda())
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    h = plan_ref.decode_header(plan.dump())
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), h


def _cascade_mixed():
    w = workloads.make_custom("cas", [30, 1, 4, 200, 1, 8, 1], [300, 500, 600, 900, 70, 400, 200], 16, 2,
                              128, 16, dtype=torch.bfloat16, seed=51, permute_pages=False)
    ind, ptr = w.kv_page_indices.copy(), w.kv_page_indptr
    for b in (1, 2):
        ind[ptr[b]:ptr[b] + 10] = ind[ptr[0]:ptr[0] + 10]
    ind[ptr[4]:ptr[4] + 4] = ind[ptr[3]:ptr[3] + 4]
    w.kv_page_indices = ind
    return w, [0, 3, 5, 7], [10, 4, 0]


def test_cascade_prefix_workload():
    """The prefix batch (64 requests appending 30 tokens to a 200-token
    prompt whose first 12 pages are shared) planned as a cascade: the
    shared 192 keys are attended once for all 1920 query tokens."""
    w = workloads.prefix()
    groups, args = workloads.split_prefix(w, [0, 64], [12])
    out, lse, h = _cascade_run(w, groups, args)
    assert h["n_groups"] == 1
    ro, rl = A.attention(w)
    assert_close(out, lse, ro, rl, w.dtype, what="cascade prefix")
    o2, l2, _ = run(w)
    assert np.allclose(out, o2, atol=1e-2, rtol=0) and np.allclose(lse, l2, atol=1e-3, rtol=0)


@pytest.mark.parametrize("opts", [{}, {"prefill_chunk_tiles": 1, "decode_chunk_pages": 3},
                                  {"decode_cuda_cores": True}, {"kv_layout": "HND"}])
def test_cascade_mixed_groups(opts):
    """Groups of prefill, decode and few-token requests behind 10- and
    4-page prefixes, and a group without one, against the oracle on the
    flattened page tables."""
    w, gind, npre = _cascade_mixed()
    groups, args = workloads.split_prefix(w, gind, npre)
    kv = w.kv_cache.permute(0, 1, 3, 2, 4).contiguous() if opts.get("kv_layout") == "HND" else None
    out, lse, h = _cascade_run(w, groups, args, kv=kv, **opts)
    assert h["n_groups"] == 3
    ro, rl = A.attention(w)
    assert_close(out, lse, ro, rl, w.dtype, what=f"cascade {opts}")


@pytest.mark.parametrize("cuda_cores", [False, True])
def test_cascade_shared_prefix_decode(cuda_cores):
    """One-token decodes continuing one long shared prompt, as a cascade:
    the prompt's attention is one prefill over all the decodes' query rows."""
    w = workloads.prefix_decode(batch_size=24, prefix_len=1024, own_lo=30, own_hi=300)
    groups, args = workloads.split_prefix(w, [0, 24], [64])
    out, lse, h = _cascade_run(w, groups, args, decode_cuda_cores=cuda_cores)
    assert h["n_groups"] == 1 and h["n_pre"] > 0 and h["n_dec"] > 0
    ro, rl = A.attention(w)
    assert_close(out, lse, ro, rl, w.dtype, what="cascade decode")


# ---------------------------------------------------------------- failure handling and host threads


@pytest.mark.parametrize("name,opts", [
    ("tiny", {}), ("tiny", {"force_prefill": True}), ("tiny", {"force_prefill": True, "prefill_q_tiles": 1}),
    ("tiny", {"force_cp_async": True, "force_prefill": True}),
    ("decode", {"decode_chunk_pages": 64}), ("decode", {"decode_cuda_cores": True, "decode_chunk_pages": 64})])
def test_wait_limit_gives_up_then_normal_run(name, opts):
    """Every in-kernel pipeline wait is bounded.  The wait_limit_cycles test
    hook cuts the bound to one clock cycle and has one thread of every CTA
    wait on a barrier that nothing completes (a flag nobody sets): that wait
    gives up, the CTA drains the copies and MMAs it has in flight, releases
    its TMEM and returns, and the run reports PA_DEV_TIMEOUT through the
    device status word.  A normal run on the same workspace afterwards
    matches the oracle."""
    w = workloads.tiny() if name == "tiny" else workloads.decode(batch_size=16, seq_len=1000)
    ws = torch.empty(pa.DEFAULT_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
    q, kv = w.q.cuda(), w.kv_cache.cuda()
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype, workspace=ws, wait_limit_cycles=1, **opts)
    plan.run(q, kv)
    torch.cuda.synchronize()
    flags = plan.device_status()
    assert flags & pa.PA_DEV_TIMEOUT, f"no wait gave up (flags {flags})"
    plan.close()
    ro, rl = A.attention(w)
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype, workspace=ws, **opts)
    out, lse = plan.run(q, kv)
    torch.cuda.synchronize()
    assert plan.device_status() == 0, pa.last_error()
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, w.dtype,
                 what=f"after a timed-out run {opts}")


def test_host_threads():
    """Host threads: (a) two threads, each with its own plan, workspace and
    stream, run at the same time; (b) two threads run one plan on one shared
    stream, each alternating between two copies of the cache, so that the
    plan's cached TMA descriptors are re-made on almost every call.  Every
    result matches the oracle."""
    import threading
    wa = workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    wb = workloads.ragged()
    refs = {id(w): A.attention(w) for w in (wa, wb)}
    errors = []

    def own_plan(w, reps):
        try:
            st = torch.cuda.Stream()
            q, kv = w.q.cuda(), w.kv_cache.cuda()
            torch.cuda.synchronize()
            plan = pa.Plan(**w.plan_args(), dtype=w.dtype, stream=st)
            outs = []
            for _ in range(reps):
                outs.append(plan.run(q, kv, stream=st))
            st.synchronize()
            assert plan.device_status(stream=st) == 0
            ro, rl = refs[id(w)]
            for out, lse in outs:
                assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, w.dtype,
                             what="own plan, own thread")
        except Exception as e:  # reported by the main thread
            errors.append(e)

    ts = [threading.Thread(target=own_plan, args=(w, 6)) for w in (wa, wb)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors

    w = wa
    st = torch.cuda.Stream()
    q = w.q.cuda()
    kvs = [w.kv_cache.cuda(), w.kv_cache.cuda()]
    torch.cuda.synchronize()
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype, stream=st)
    results = {0: [], 1: []}

    def shared_plan(k):
        try:
            for i in range(8):
                results[k].append(plan.run(q, kvs[(i + k) % 2], stream=st))
        except Exception as e:
            errors.append(e)

    ts = [threading.Thread(target=shared_plan, args=(k,)) for k in (0, 1)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    st.synchronize()
    assert not errors, errors
    assert plan.device_status(stream=st) == 0
    ro, rl = refs[id(w)]
    first = results[0][0][0].cpu()
    for k in (0, 1):
        for out, lse in results[k]:
            assert torch.equal(out.cpu(), first)
    out, lse = results[1][-1]
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, w.dtype, what="shared plan")


@pytest.mark.parametrize("G", [2, 8])
def test_decode_cp_async_equals_tma(G):
    """Decode staged by cp.async (force_cp_async) writes the same shared-memory
    tiles as the TMA path, so the outputs are identical bit for bit; both
    match the oracle."""
    w = workloads.make_custom("dcp", [1] * 9, [1, 15, 16, 17, 300, 1000, 64, 129, 2000], 2 * G, 2, 128, 16,
                              dtype=torch.bfloat16, seed=G)
    ro, rl = A.attention(w)
    o1, l1, _ = run(w, decode_chunk_pages=8)
    o2, l2, _ = run(w, decode_chunk_pages=8, force_cp_async=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert_close(o1, l1, ro, rl, w.dtype, what=f"decode G{G}")


def _remap_pages(w, sigma):
    """The same logical cache with physical page i moved to sigma[i]."""
    sigma = np.asarray(sigma, np.int64)
    cache = torch.empty_like(w.kv_cache)
    cache[torch.from_numpy(sigma)] = w.kv_cache
    w.kv_cache = cache
    w.kv_page_indices = sigma[w.kv_page_indices].astype(np.int32)
    return w


@pytest.mark.parametrize("ps", [8, 16, 32, 64])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_consecutive_page_runs(ps, layout):
    """Page tables whose pages are physically consecutive (as a fresh cache
    allocates them) against the same cache with page pairs swapped here and
    there: prefill, small-query and decode requests, both layouts.  Every
    output matches the oracle, and both placements give identical bits."""
    qo = [1, 1, 200, 3, 130, 1]
    kv = [1500, 64, 200, 700, 900, 2000]
    w = workloads.make_custom("runs", qo, kv, 16, 2, 128, ps, dtype=torch.bfloat16, seed=ps, permute_pages=False)
    ro, rl = A.attention(w)
    kvd = _hnd(w.kv_cache) if layout == "HND" else None
    o1, l1, _ = run(w, kv=kvd, kv_layout=layout, decode_chunk_pages=max(1, 256 // ps))
    assert_close(o1, l1, ro, rl, w.dtype, what=f"contiguous pages ps {ps} {layout}")
    sigma = np.arange(w.num_pages)
    for i in range(3, w.num_pages - 1, 7):   # swap pairs: every run of a stage or tile is broken somewhere
        sigma[i], sigma[i + 1] = sigma[i + 1], sigma[i]
    w2 = _remap_pages(w, sigma)
    kvd = _hnd(w2.kv_cache) if layout == "HND" else None
    o2, l2, _ = run(w2, kv=kvd, kv_layout=layout, decode_chunk_pages=max(1, 256 // ps))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("G,qo", [(8, 1), (4, 2), (1, 5), (8, 4), (16, 1)],
                         ids=["rows8_G8", "rows8_G4", "rows5_G1", "rows32", "rows16"])
@pytest.mark.parametrize("ps", [16, 4])
def test_decode_launch_shapes_agree(G, qo, ps):
    """The same small-query items launched one CTA per SM (six stages, more
    producer warps) and two CTAs per SM (three stages): planned for many SMs
    and for four, with the decode split fixed so that the items agree.  The
    outputs are identical bit for bit and match the oracle (row classes 0, 1
    and 2; TMA and cp.async staging)."""
    qos = [qo] * 12
    kvs = [qo + 130 + 97 * i for i in range(12)]
    w = workloads.make_custom("shape", qos, kvs, 2 * G, 2, 128, ps, dtype=torch.bfloat16, seed=G * 10 + qo)
    ro, rl = A.attention(w)
    chunk = max(1, 128 // ps)
    o1, l1, p1 = run(w, num_sms=1024, decode_chunk_pages=chunk)
    o2, l2, p2 = run(w, num_sms=4, decode_chunk_pages=chunk)
    h1, h2 = plan_ref.decode_header(p1.dump()), plan_ref.decode_header(p2.dump())
    assert h1["n_pre"] == 0 and h1["n_dec"] == h2["n_dec"] and h1["n_dec"] > 4
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert_close(o1, l1, ro, rl, w.dtype, what=f"launch shapes G{G} qo{qo} ps{ps}")


def test_back_to_back_runs_chain():
    """Runs queued back to back on one stream, whose kernels may start before
    the previous kernel ends (programmatic dependent launch): run 2 reads as
    its q the out that run 1 writes; run 4 overwrites that buffer right after
    run 2 and a copy have read it; all runs share the plan's split-KV
    partial states.  Every result equals the same run made after a full
    device synchronisation, bit for bit."""
    w = workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype)
    q, kv = w.q.cuda(), w.kv_cache.cuda()
    q3 = (w.q * 0.5).cuda()
    o1, _ = plan.run(q, kv)
    o2, _ = plan.run(o1, kv)
    o3, _ = plan.run(q3, kv)
    o1b = o1.clone()
    o4, _ = plan.run(q3, kv, out=o1)     # overwrites o1 right after the clone reads it
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    r1, _ = plan.run(q, kv)
    torch.cuda.synchronize()
    r2, _ = plan.run(r1.clone(), kv)
    torch.cuda.synchronize()
    r3, _ = plan.run(q3, kv)
    torch.cuda.synchronize()
    assert torch.equal(o1b, r1)
    assert torch.equal(o2, r2)
    assert torch.equal(o3, r3) and torch.equal(o1, r3) and torch.equal(o4, r3)


@pytest.mark.parametrize("G", [1, 4, 16])
@pytest.mark.parametrize("q_tiles", [1, 2])
def test_output_tiles_every_fill(G, q_tiles):
    """Prefill output tiles filled to every row count the epilogue treats
    apart: fewer than 32 valid rows (written row by row), whole 32-row boxes
    plus a remainder, and full 128-row tiles (TMA stores), in tile A and in
    tile B of two-tile items; each against the oracle."""
    tq = 128 // G
    qos = sorted({max(1, n) for n in (tq // 4 - 1, tq // 4, tq // 4 + 1, tq // 2, 3 * tq // 4 + 1, tq - 1, tq,
                                      tq + 1, tq + tq // 4, 2 * tq - 1, 2 * tq)})
    kvs = [q + 70 for q in qos]
    w = workloads.make_custom("fill", qos, kvs, 2 * G, 2, 128, 16, dtype=torch.bfloat16, seed=G + q_tiles)
    ro, rl = A.attention(w)
    out, lse, plan = run(w, prefill_q_tiles=q_tiles, force_prefill=True)
    assert plan_ref.decode_header(plan.dump())["n_pre"] > 0
    assert_close(out, lse, ro, rl, w.dtype, what=f"output tiles G{G} q_tiles {q_tiles}")
