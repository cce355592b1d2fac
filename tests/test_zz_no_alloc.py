"""pagedattn_run_decode_noalloc, the decode entry point that allocates no
device memory.

It serves callers that cannot call cudaMalloc: serving processes that keep
all free GPU memory reserved for their KV cache, and latency-critical code
that must not call cudaFree because it synchronises the device.  Instead of
a caller workspace it keeps the plan metadata and the split-KV partial
states in a fixed array inside the library.  This test calls it through the
C ABI twice in a row, on two different decode batches that both need splits
(so the second call runs over what the first left in the array), and checks
each output against the ordinary pagedattn_run path within the tolerance of
the other parity tests.  It lives in its own file, collected last.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

pa = pytest.importorskip("attention_paged_kv_gb300")
from parity import LSE_TOL, out_tol  # noqa: E402


def _batches():
    a = workloads.decode(batch_size=48, seq_len=1000)                 # fp16, 8 query heads per kv head
    lens = workloads.randint_incl(1, 3000, 40, 2024).tolist()
    b = workloads.make_custom("noalloc_b", [1] * 40, lens, 16, 4, 128, 16, dtype=torch.bfloat16, seed=91)
    return [(a, 4), (b, 3)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_decode_matches_run_two_calls_in_a_row():
    lib = pa.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.current_stream()
    for w, chunk in _batches():
        q, kv = w.q.cuda(), w.kv_cache.cuda()
        ref_plan = pa.Plan(**w.plan_args(), dtype=w.dtype, decode_chunk_pages=chunk)
        ref_out, ref_lse = ref_plan.run(q, kv)
        host_plan = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=sms,
                            decode_chunk_pages=chunk)
        hdr = host_plan.dump()
        assert hdr[13] == 0 and hdr[14] > 0, "expected a decode-only batch with split requests"
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = lib.pagedattn_run_decode_noalloc(host_plan._h, q.data_ptr(), kv.data_ptr(), out.data_ptr(),
                                              lse.data_ptr(), stream.cuda_stream)
        assert st == pa.PA_OK, pa.last_error()
        torch.cuda.synchronize()
        ro = ref_out.double().cpu().numpy()
        go = out.double().cpu().numpy()
        assert np.isfinite(go).all()
        assert (np.abs(go - ro) <= out_tol(ro, w.dtype)).all()
        assert (np.abs(lse.double().cpu().numpy() - ref_lse.double().cpu().numpy()) <= LSE_TOL).all()


def test_noalloc_rejects_prefill_batches():
    lib = pa.load()
    w = workloads.make_custom("pre", [1, 40], [9, 300], 16, 2, 128, 16, seed=3)  # 40 x 8 rows: prefill
    plan = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=148)
    assert plan.dump()[13] > 0
    st = lib.pagedattn_run_decode_noalloc(plan._h, None, None, None, None, None)
    assert st == pa.PA_ERR_UNSUPPORTED and "decode" in pa.last_error()
