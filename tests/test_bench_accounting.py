"""bench.py's algorithmic accounting splits a batch into the prefill and the
decode part by the planner's rule; the split must agree with the plan the
library builds (host-only plans, no GPU)."""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402
from oracle import plan_ref  # noqa: E402

pa = pytest.importorskip("attention_paged_kv_gb300")

QOS = [1, 300, 1, 5, 130, 2, 4, 0]
KVS = [1, 300, 700, 400, 900, 600, 100, 9]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_accounting_split_matches_the_plan(D, G):
    w = workloads.make_custom("acc", QOS, KVS, 2 * G, 2, D, 16, dtype=torch.bfloat16, seed=G + D)
    acc = bench.accounting(w)
    p = pa.Plan(**w.plan_args(), dtype=w.dtype, host_only=True, num_sms=148)
    try:
        dec, pre, _ = plan_ref.items(p.dump())
    finally:
        p.close()
    qo = np.diff(w.qo_indptr)
    dec_reqs = sorted({int(b) for b in dec[:, 0]})
    pre_reqs = sorted({int(b) for b in pre[:, 0]})
    assert not set(dec_reqs) & set(pre_reqs)
    assert acc["decode"]["rows"] == int(qo[dec_reqs].sum())
    assert acc["prefill"]["rows"] == int(qo[pre_reqs].sum())
