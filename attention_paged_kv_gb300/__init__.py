"""Batched ragged attention over a paged KV cache for one GB300 (sm_103a).

The computation runs in ``libpagedattn.so`` (C ABI, include/pagedattn.h):
a tcgen05/TMEM tensor-core prefill kernel, a warp-MMA small-query kernel
(decode and few-token requests), a CUDA-core decode kernel, a split-state
merge kernel and a C++ planner.  This package is the
thin ctypes binding with the same names.  Build the library with
``python -m attention_paged_kv_gb300.build``.
"""
from ._binding import (DEFAULT_WORKSPACE_BYTES, EXPORTED, PA_BF16, PA_DEV_BAD_INDEX, PA_DEV_TIMEOUT,
                       PA_ERR_CUDA, PA_ERR_DEVICE_CHECK, PA_ERR_INVALID_ARG, PA_ERR_TIMEOUT,
                       PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE_TOO_SMALL, PA_FP16, PA_OK, PA_STAGE_ALL,
                       PA_STAGE_DECODE, PA_STAGE_MERGE, PA_STAGE_PREFILL, PA_LAYOUT_HND, PA_LAYOUT_NHD,
                       LIB_PATH, Options,
                       PagedAttnError, Plan, check, last_error, load, version, workspace_size)

__all__ = ["Plan", "PagedAttnError", "workspace_size", "load", "version", "last_error", "check", "Options",
           "EXPORTED", "LIB_PATH", "DEFAULT_WORKSPACE_BYTES"]
