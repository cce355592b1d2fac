"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, plans bit-for-bit like the restated rules, and rejects bad input
with the documented status codes.  No GPU is needed."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import workloads
from oracle import plan_ref

pa = pytest.importorskip("attention_paged_kv_gb300")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pa.LIB_PATH):
        from attention_paged_kv_gb300 import build
        build.build()
    return pa.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "pagedattn.h")).read()
    return sorted(set(re.findall(r"PAGEDATTN_API\s+[\w\s\*]+?\b(pagedattn_\w+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    decl = declared_symbols()
    assert len(decl) >= 10
    assert sorted(decl) == sorted(pa.EXPORTED)
    for name in decl:
        assert hasattr(lib, name), name
    assert pa.version() == "0.2.0"


def _ref(w, **kw):
    args = w.plan_args()
    return plan_ref.build(**args, dtype=plan_ref.FP16 if w.dtype == torch.float16 else plan_ref.BF16, **kw)


def _lib_blob(w, **kw):
    p = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, **kw)
    try:
        return p.dump()
    finally:
        p.close()


CASES = [
    ("tiny", {}), ("tiny", {"force_prefill": True}), ("tiny", {"prefill_chunk_tiles": 1}),
    ("decode", {}), ("decode", {"decode_chunk_pages": 3}), ("ragged", {}), ("ragged_padded", {}),
    ("prefix", {}), ("prefix_dup", {}), ("mixed_small", {}), ("mixed_small", {"prefill_chunk_tiles": 2}),
    ("random", {}), ("random_nc", {}), ("empty", {}), ("qo0", {}),
    ("random", {"decode_cuda_cores": True}), ("smallq", {}), ("smallq", {"decode_cuda_cores": True}),
    ("smallq", {"decode_chunk_pages": 2}), ("smallq_g16", {}), ("smallq_g1", {}), ("specdec", {}),
    ("tiny", {"kv_layout": "HND"}), ("smallq", {"kv_layout": "HND"}),
    ("d256", {}), ("d256", {"prefill_chunk_tiles": 1, "decode_chunk_pages": 2}), ("d256_g16", {}),
    ("ragged", {"prefill_q_tiles": 1}), ("tiny", {"prefill_q_tiles": 1}), ("mixed_small", {"prefill_q_tiles": 2}),
]


def make(name):
    if name == "tiny":
        return workloads.tiny()
    if name == "decode":
        return workloads.decode()
    if name == "ragged":
        return workloads.ragged()
    if name == "ragged_padded":
        return workloads.ragged(padded=True)
    if name == "prefix":
        return workloads.prefix()
    if name == "prefix_dup":
        return workloads.prefix(duplicated=True)
    if name == "mixed_small":
        return workloads.mixed(num_decode=24, prefill_len=700, kv_lo=16, kv_hi=3000)
    if name == "random":
        return workloads.make_custom("r", [1, 5, 0, 130, 1, 64], [9, 300, 4, 130, 2500, 64], 16, 4, 128, 8,
                                     dtype=torch.bfloat16, seed=5)
    if name == "random_nc":
        return workloads.make_custom("r", [3, 1, 200], [2, 7, 40], 8, 8, 64, 2, causal=False, seed=6)
    if name == "smallq":  # G 8: 32, 32, 16 and 8 packed rows, 64 rows and a 9-token prefill
        return workloads.make_custom("sq", [4, 4, 2, 1, 8, 9], [300, 40, 900, 70, 500, 9], 16, 2, 128, 16,
                                     dtype=torch.bfloat16, seed=11)
    if name == "smallq_g16":
        return workloads.make_custom("sq16", [1, 2, 4, 5], [77, 500, 260, 30], 16, 1, 64, 8, seed=12)
    if name == "smallq_g1":
        return workloads.make_custom("sq1", [64, 65, 3, 1], [64, 200, 1000, 9], 2, 2, 64, 4, seed=13)
    if name == "specdec":
        return workloads.mixed(num_decode=24, prefill_len=0, kv_lo=16, kv_hi=3000, decode_qo=4)
    if name == "d256":  # G 4: decodes, a 5-token request, prefills of 1 and 3 tiles
        return workloads.make_custom("d256", [1, 300, 1, 5, 130, 0], [1, 300, 700, 400, 900, 17], 8, 2, 256, 16,
                                     seed=14)
    if name == "d256_g16":
        return workloads.make_custom("d256g", [1, 1, 9], [70, 500, 900], 16, 1, 256, 8, dtype=torch.bfloat16,
                                     seed=15)
    if name == "empty":
        return workloads.make_custom("e", [], [], 4, 1, 64, 16, seed=7)
    if name == "qo0":
        return workloads.make_custom("z", [0, 2, 0], [5, 3, 17], 4, 2, 128, 4, seed=8)
    raise KeyError(name)


@pytest.mark.parametrize("name,kw", CASES, ids=[f"{n}-{'-'.join(f'{k}{v}' for k, v in kw.items())}" for n, kw in CASES])
@pytest.mark.parametrize("sms", [148, 7])
def test_plan_bit_exact_vs_restated_rules(lib, name, kw, sms):
    w = make(name)
    got = _lib_blob(w, num_sms=sms, **kw)
    want = _ref(w, num_sms=sms, **kw)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_plan_default_num_sms_needs_device(lib):
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    w = workloads.tiny()
    with pytest.raises(pa.PagedAttnError) as e:
        pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def _expect(status, w, **over):
    args = w.plan_args()
    args.update({k: v for k, v in over.items() if k in args})
    kw = {k: v for k, v in over.items() if k not in args}
    kw.setdefault("num_sms", 148)
    dtype = kw.pop("dtype", w.dtype)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.Plan(**args, dtype=dtype, host_only=True, **kw)
    assert e.value.status == status, str(e.value)
    assert pa.last_error()


def test_errors_invalid(lib):
    w = workloads.tiny()
    _expect(pa.PA_ERR_INVALID_ARG, w, qo_indptr=np.array([1, 2, 5, 10, 18]))
    _expect(pa.PA_ERR_INVALID_ARG, w, qo_indptr=np.array([0, 3, 2, 9, 17]))
    _expect(pa.PA_ERR_INVALID_ARG, w, kv_page_indptr=np.array([0, 2, 1, 11, 17]))
    # the timing script's literal last page length, seq_length % page_size = 0
    _expect(pa.PA_ERR_INVALID_ARG, w, kv_last_page_len=np.array([4, 0, 1, 4]))
    _expect(pa.PA_ERR_INVALID_ARG, w, kv_last_page_len=np.array([4, 5, 1, 4]))
    bad = w.kv_page_indices.copy()
    bad[3] = w.num_pages
    _expect(pa.PA_ERR_INVALID_ARG, w, kv_page_indices=bad)
    bad[3] = -1
    _expect(pa.PA_ERR_INVALID_ARG, w, kv_page_indices=bad)
    _expect(pa.PA_ERR_INVALID_ARG, w, num_qo_heads=3, num_kv_heads=2)
    # causal: more query rows than keys
    _expect(pa.PA_ERR_INVALID_ARG, w, qo_indptr=np.array([0, 9, 12, 17, 25]))


def test_errors_unsupported(lib):
    w = workloads.tiny()
    _expect(pa.PA_ERR_UNSUPPORTED, w, head_dim=96)
    _expect(pa.PA_ERR_UNSUPPORTED, w, head_dim=512)
    _expect(pa.PA_ERR_INVALID_ARG, w, prefill_q_tiles=3)
    _expect(pa.PA_ERR_UNSUPPORTED, make("d256"), prefill_q_tiles=2)
    _expect(pa.PA_ERR_UNSUPPORTED, w, page_size=3)
    _expect(pa.PA_ERR_UNSUPPORTED, w, page_size=256)
    _expect(pa.PA_ERR_UNSUPPORTED, w, num_qo_heads=6, num_kv_heads=2)   # group 3 does not divide 128
    args = w.plan_args()
    a = [np.ascontiguousarray(np.asarray(args[k], np.int32)) for k in
         ("qo_indptr", "kv_page_indptr", "kv_page_indices", "kv_last_page_len")]
    h = ctypes.c_void_p(0)
    o = pa.Options()
    o.num_sms = 148
    P = ctypes.POINTER(ctypes.c_int32)
    st = lib.pagedattn_plan(*[x.ctypes.data_as(P) for x in a], 4, 2, 1, 64, 4, w.num_pages, 7, 1, None, 0,
                            ctypes.byref(o), None, ctypes.byref(h))
    assert st == pa.PA_ERR_UNSUPPORTED


def test_workspace_too_small_and_options(lib):
    w = workloads.tiny()
    args = w.plan_args()
    a = [np.ascontiguousarray(np.asarray(args[k], np.int32)) for k in
         ("qo_indptr", "kv_page_indptr", "kv_page_indices", "kv_last_page_len")]
    P = ctypes.POINTER(ctypes.c_int32)
    h = ctypes.c_void_p(0)
    o = pa.Options()
    o.num_sms = 148
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    st = lib.pagedattn_plan(*[x.ctypes.data_as(P) for x in a], 4, 2, 1, 64, 4, w.num_pages, 0, 1, fake, 64,
                            ctypes.byref(o), None, ctypes.byref(h))
    assert st == pa.PA_ERR_WORKSPACE_TOO_SMALL and not h.value
    o.reserved[0] = 3
    st = lib.pagedattn_plan(*[x.ctypes.data_as(P) for x in a], 4, 2, 1, 64, 4, w.num_pages, 0, 1, None, 0,
                            ctypes.byref(o), None, ctypes.byref(h))
    assert st == pa.PA_ERR_INVALID_ARG
    o.reserved[0] = 0
    o.kv_layout = 2
    st = lib.pagedattn_plan(*[x.ctypes.data_as(P) for x in a], 4, 2, 1, 64, 4, w.num_pages, 0, 1, None, 0,
                            ctypes.byref(o), None, ctypes.byref(h))
    assert st == pa.PA_ERR_UNSUPPORTED and "kv_layout" in pa.last_error()
    n = pa.workspace_size(**args, dtype=w.dtype, num_sms=148)
    assert n == plan_ref.decode_header(_ref(w, num_sms=148))["total_bytes"]


def test_host_only_plan_cannot_run(lib):
    w = workloads.tiny()
    p = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=148)
    st = lib.pagedattn_run(p._h, None, None, None, None, None)
    assert st == pa.PA_ERR_INVALID_ARG
    assert lib.pagedattn_plan_destroy(None) == pa.PA_OK
    p.close()


def test_plan_metadata_semantics(lib):
    """The decode script's batch runs unsplit on 148 SMs (128 items: one
    wave that covers most SMs) and in splits of 256 keys on 256 SMs; the
    mixed batch keeps its long prefill unsplit."""
    w = workloads.decode()
    h = plan_ref.decode_header(_lib_blob(w, num_sms=148))
    assert (h["n_dec"], h["n_pre"], h["n_merge"], h["dec_chunk_pages"]) == (128, 0, 0, 128)
    h = plan_ref.decode_header(_lib_blob(w, num_sms=256))
    assert (h["n_dec"], h["n_pre"], h["n_merge"], h["dec_chunk_pages"]) == (512, 0, 128, 16)
    w = workloads.mixed(num_decode=8, prefill_len=8192, kv_lo=512, kv_hi=8192)
    blob = _lib_blob(w, num_sms=148)
    dec, pre, mer = plan_ref.items(blob)
    assert (pre[:, 6] == -1).all()                 # no prefill split
    assert pre[:, 3].max() == 32                   # 32 tokens x 8 heads per item (two tiles)
    assert pre[0, 5] - pre[0, 4] == 8192           # longest first


def test_plan_small_query_semantics(lib):
    """Requests of a few query tokens (qo_len * G <= 32 packed rows) become
    small-query items of the decode kernels, grouped by row class; their
    split groups merge per (token, kv head) with a stride of qo_len * G."""
    w = workloads.mixed(num_decode=24, prefill_len=0, kv_lo=200, kv_hi=3000, decode_qo=4)
    blob = _lib_blob(w, num_sms=148, decode_chunk_pages=16)
    h = plan_ref.decode_header(blob)
    dec, pre, mer = plan_ref.items(blob)
    assert h["n_pre"] == 0 and h["dec_cuda_cores"] == 0
    assert h["dec_class_items"] == [0, 0, h["n_dec"], 0]   # 4 tokens x 8 heads = 32 rows
    split = dec[dec[:, 4] >= 0]
    assert len(split) and (mer[:, 3] == 32).all()
    assert len(mer) == 4 * len({(int(b), int(k)) for b, k in split[:, :2]})
    # the option keeps multi-token requests on the prefill kernel
    h2 = plan_ref.decode_header(_lib_blob(w, num_sms=148, decode_cuda_cores=True))
    assert h2["n_dec"] == 0 and h2["dec_cuda_cores"] == 1
    # G <= 2 with single-token requests only: CUDA cores; one two-token request moves all to MMA
    a = workloads.make_custom("g2", [1, 1, 1], [10, 20, 30], 4, 2, 64, 4, seed=1)
    assert plan_ref.decode_header(_lib_blob(a, num_sms=148))["dec_cuda_cores"] == 1
    b = workloads.make_custom("g2", [1, 2, 1], [10, 200, 30], 4, 2, 64, 4, seed=1)
    c = workloads.make_custom("g2", [1, 2, 1], [10, 20, 30], 4, 2, 64, 4, seed=1)  # 2 tokens, 20 keys: prefill
    hc = plan_ref.decode_header(_lib_blob(c, num_sms=148))
    assert hc["dec_cuda_cores"] == 1 and hc["n_pre"] > 0
    hb = plan_ref.decode_header(_lib_blob(b, num_sms=148))
    assert hb["dec_cuda_cores"] == 0 and hb["n_pre"] == 0 and hb["dec_class_items"][0] == hb["n_dec"]


def test_plan_head_dim_256_semantics(lib):
    """At head_dim 256 a prefill item is one 128-row tile, single-token
    requests at G <= 8 decode on the CUDA-core kernel, and every other
    request (several tokens, or G = 16) goes to the prefill kernel."""
    w = make("d256")
    blob = _lib_blob(w, num_sms=148)
    h = plan_ref.decode_header(blob)
    dec, pre, mer = plan_ref.items(blob)
    assert h["dec_cuda_cores"] == 1
    assert sorted({int(b) for b in dec[:, 0]}) == [0, 2]          # the two single-token requests
    assert sorted({int(b) for b in pre[:, 0]}) == [1, 3, 4]       # 5 tokens, 300 and 130 tokens
    assert pre[:, 3].max() == 32                                  # 32 tokens x 4 heads = one tile
    r1 = pre[pre[:, 0] == 1]
    assert len(r1) == 2 * 10 and (r1[:, 3] == 32).sum() == 2 * 9  # 300 tokens: 9 tiles of 32 and one of 12, x 2 kv heads
    g16 = plan_ref.decode_header(_lib_blob(make("d256_g16"), num_sms=148))
    assert g16["n_dec"] == 0 and g16["n_pre"] > 0


def test_plan_one_tile_rule(lib):
    """Prefill items of one 128-row tile when most two-tile items would run
    only their first tile (2 n1 <= 3 n2 with n1, n2 the item counts at 128
    and 256 rows): the prefix batch (30 tokens x G 4 = 120 rows a request)
    and the tiny batch take one tile, the ragged and mixed batches two; the
    option overrides the rule, and head_dim 256 always takes one."""
    def tiles(w, **kw):
        return plan_ref.decode_header(_lib_blob(w, num_sms=148, **kw))["pre_tiles"]
    assert tiles(workloads.prefix()) == 1 and tiles(workloads.tiny()) == 1
    assert tiles(workloads.ragged()) == 2 and tiles(make("mixed_small")) == 2
    assert tiles(workloads.ragged(), prefill_q_tiles=1) == 1 and tiles(workloads.prefix(), prefill_q_tiles=2) == 2
    assert tiles(make("d256")) == 1
    # the rule at its edge: G 4 (32 tokens a tile), one request of 64 tokens -> n1 2, n2 1: two tiles;
    # two requests of 32 -> n1 2, n2 2: one tile
    a = workloads.make_custom("e1", [64], [64], 8, 2, 128, 16, seed=1)
    b = workloads.make_custom("e2", [32, 32], [32, 32], 8, 2, 128, 16, seed=1)
    assert tiles(a) == 2 and tiles(b) == 1


def _cascade_cases():
    """(name, workload, group_indptr, prefix pages per group)."""
    pre = workloads.prefix()                                    # 64 requests share 12 full pages
    mixed = workloads.make_custom("cas", [30, 1, 4, 200, 1, 8, 1], [300, 500, 600, 900, 70, 400, 200], 16, 2,
                                  128, 16, dtype=torch.bfloat16, seed=51, permute_pages=False)
    # give requests 0-2 a common 10-page prefix and requests 3-4 a common 4-page one (tables rewritten)
    ind = mixed.kv_page_indices.copy()
    ptr = mixed.kv_page_indptr
    for b in (1, 2):
        ind[ptr[b]:ptr[b] + 10] = ind[ptr[0]:ptr[0] + 10]
    ind[ptr[4]:ptr[4] + 4] = ind[ptr[3]:ptr[3] + 4]
    mixed.kv_page_indices = ind
    return [("prefix", pre, [0, 64], [12]), ("mixed", mixed, [0, 3, 5, 7], [10, 4, 0])]


@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("kw", [{}, {"prefill_chunk_tiles": 1, "decode_chunk_pages": 3}, {"decode_cuda_cores": True}])
def test_cascade_plan_bit_exact_vs_restated_rules(lib, case, kw):
    name, w, gind, npre = _cascade_cases()[case]
    groups, args = workloads.split_prefix(w, gind, npre)
    dt = plan_ref.FP16 if w.dtype == torch.float16 else plan_ref.BF16
    want = plan_ref.build(**args, dtype=dt, num_sms=148, prefix_groups=groups, **kw)
    p = pa.Plan(**args, dtype=w.dtype, host_only=True, num_sms=148, prefix_groups=groups, **kw)
    got = p.dump()
    p.close()
    assert got.shape == want.shape and np.array_equal(got, want)
    h = plan_ref.decode_header(got)
    assert h["n_groups"] == len(gind) - 1 and h["n_pre"] > 0
    n = pa.workspace_size(**args, dtype=w.dtype, num_sms=148, prefix_groups=groups, **kw)
    assert n == h["total_bytes"]


def test_cascade_plan_errors(lib):
    name, w, gind, npre = _cascade_cases()[1]
    groups, args = workloads.split_prefix(w, gind, npre)
    bad = (np.array([0, 3, 6], np.int32), groups[1][:3], groups[2])      # groups end before batch_size
    with pytest.raises(pa.PagedAttnError) as e:
        pa.Plan(**args, dtype=w.dtype, host_only=True, num_sms=148, prefix_groups=bad)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    badp = groups[2].copy()
    badp[0] = w.num_pages
    with pytest.raises(pa.PagedAttnError) as e:
        pa.Plan(**args, dtype=w.dtype, host_only=True, num_sms=148, prefix_groups=(groups[0], groups[1], badp))
    assert e.value.status == pa.PA_ERR_INVALID_ARG
