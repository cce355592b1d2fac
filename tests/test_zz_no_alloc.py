"""pagedattn_run_decode_noalloc, the decode entry point that allocates no
device memory.

It serves callers that cannot call cudaMalloc: serving processes that keep
all free GPU memory reserved for their KV cache, and latency-critical code
that must not call cudaFree because it synchronises the device.  Instead of
a caller workspace it keeps the plan metadata and the split-KV partial
states in a fixed array inside the library.  These tests call it through
the C ABI several times in a row on decode batches that need splits (so
every call runs over what the last one left in the array) and check each
output against the ordinary pagedattn_run path and against the fp64 oracle,
within the tolerance of the other parity tests, and read the array's status
word back after every call.  The file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A

pytestmark = pytest.mark.gpu

pa = pytest.importorskip("attention_paged_kv_gb300")
from parity import LSE_TOL, assert_close, out_tol  # noqa: E402


def _batches():
    a = workloads.decode(batch_size=48, seq_len=1000)                 # fp16, 8 query heads per kv head
    lens = workloads.randint_incl(1, 3000, 40, 2024).tolist()
    b = workloads.make_custom("noalloc_b", [1] * 40, lens, 16, 4, 128, 16, dtype=torch.bfloat16, seed=91)
    return [(a, 4), (b, 3)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _noalloc(lib, w, chunk, stream, **opts):
    """Plan host-only, run through the no-alloc entry point, read its status
    word back; returns (out, lse) on the device."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q, kv = w.q.cuda(), w.kv_cache.cuda()
    if opts.get("kv_layout") == "HND":
        kv = kv.permute(0, 1, 3, 2, 4).contiguous()
    host_plan = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=sms,
                        decode_chunk_pages=chunk, **opts)
    hdr = host_plan.dump()
    assert hdr[13] == 0 and hdr[14] > 0, "expected a decode-only batch with split requests"
    T, Hq, D = w.q.shape
    out = torch.full((T, Hq, D), float("nan"), dtype=w.dtype, device="cuda")
    lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = lib.pagedattn_run_decode_noalloc(host_plan._h, q.data_ptr(), kv.data_ptr(), out.data_ptr(),
                                          lse.data_ptr(), stream.cuda_stream)
    assert st == pa.PA_OK, pa.last_error()
    flags = ctypes.c_int32(-1)
    st = lib.pagedattn_noalloc_device_status(stream.cuda_stream, ctypes.byref(flags))
    assert st == pa.PA_OK and flags.value == 0, (st, flags.value, pa.last_error())
    return out, lse


def test_noalloc_decode_matches_run_two_calls_in_a_row():
    lib = pa.load()
    stream = torch.cuda.current_stream()
    for w, chunk in _batches():
        q, kv = w.q.cuda(), w.kv_cache.cuda()
        ref_plan = pa.Plan(**w.plan_args(), dtype=w.dtype, decode_chunk_pages=chunk)
        ref_out, ref_lse = ref_plan.run(q, kv)
        out, lse = _noalloc(lib, w, chunk, stream)
        torch.cuda.synchronize()
        ro = ref_out.double().cpu().numpy()
        go = out.double().cpu().numpy()
        assert np.isfinite(go).all()
        assert (np.abs(go - ro) <= out_tol(ro, w.dtype)).all()
        assert (np.abs(lse.double().cpu().numpy() - ref_lse.double().cpu().numpy()) <= LSE_TOL).all()
        oo, ol = A.attention(w)
        assert_close(go, lse.double().cpu().numpy(), oo, ol, w.dtype, what=f"no-alloc {w.name} vs oracle")


@pytest.mark.parametrize("case", ["page4_cp_async", "hnd", "head_dim_256", "cuda_cores_g2"])
def test_noalloc_paths_vs_oracle(case):
    """The no-alloc entry point on the other decode paths, splits forced,
    twice in a row, each call against the oracle: pages of 4 slots (cp.async
    staging), the HND cache layout, head_dim 256 (CUDA-core kernel), and
    groups of 2 query heads (CUDA-core kernel)."""
    lib = pa.load()
    stream = torch.cuda.current_stream()
    lens = [700, 1, 33, 1500, 260, 999]
    if case == "page4_cp_async":
        w = workloads.make_custom("na_p4", [1] * 6, lens, 16, 2, 128, 4, dtype=torch.bfloat16, seed=5)
        chunk, opts = 16, {}
    elif case == "hnd":
        w = workloads.make_custom("na_hnd", [1] * 6, lens, 16, 2, 128, 16, dtype=torch.float16, seed=6)
        chunk, opts = 4, {"kv_layout": "HND"}
    elif case == "head_dim_256":
        w = workloads.make_custom("na_256", [1] * 6, lens, 8, 2, 256, 16, dtype=torch.bfloat16, seed=7)
        chunk, opts = 4, {}
    else:
        w = workloads.make_custom("na_g2", [1] * 6, lens, 4, 2, 64, 8, dtype=torch.float16, seed=8)
        chunk, opts = 8, {}
    oo, ol = A.attention(w)
    for _ in range(2):
        out, lse = _noalloc(lib, w, chunk, stream, **opts)
        torch.cuda.synchronize()
        assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), oo, ol, w.dtype,
                     what=f"no-alloc {case}")


def test_noalloc_rejects_prefill_batches():
    lib = pa.load()
    w = workloads.make_custom("pre", [1, 40], [9, 300], 16, 2, 128, 16, seed=3)  # 40 x 8 rows: prefill
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=148)
    assert plan.dump()[13] > 0
    st = lib.pagedattn_run_decode_noalloc(plan._h, None, None, None, None, None)
    assert st == pa.PA_ERR_UNSUPPORTED and "decode" in pa.last_error()
