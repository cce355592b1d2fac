"""fp64 CPU oracle for batched ragged attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is the slow, plainly correct
statement of what the library computes.  Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  The library (``attention_paged_kv_gb300``) never
imports it and shares no code, table or helper with it.

Modules:

* ``oracle.attention`` -- the attention definition (two independent forms: a
  scalar ``walk`` over the page table and a per-group ``gather`` + matmul),
  the split-KV state merge, sampled rows for large batches, and the
  (page, slot) walk of the page table.
* ``oracle.plan_ref``  -- a restatement of the planner's partition rules that
  produces the plan metadata bit for bit.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, a library special case, invariants, brute force and planted
mistakes); none is "parity unpinned".
"""
from . import attention, plan_ref  # noqa: F401
