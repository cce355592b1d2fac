"""ctypes binding of libpagedattn (include/pagedattn.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no
fallback: if the shared library is missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedattn.so")

# status codes (pagedattn_status)
PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_CHECK = 5
PA_ERR_TIMEOUT = 6
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL", 4: "CUDA",
                5: "DEVICE_CHECK", 6: "TIMEOUT"}

PA_FP16 = 0
PA_BF16 = 1

PA_STAGE_PREFILL = 1
PA_STAGE_DECODE = 2
PA_STAGE_MERGE = 4
PA_STAGE_ALL = 7

PA_DEV_TIMEOUT = 1
PA_DEV_BAD_INDEX = 2

DEFAULT_WORKSPACE_BYTES = 128 * 1024 * 1024  # the timing script's workspace size

# every symbol include/pagedattn.h declares
EXPORTED = ("pagedattn_plan", "pagedattn_workspace_size", "pagedattn_run", "pagedattn_run_stages",
            "pagedattn_plan_destroy", "pagedattn_last_error", "pagedattn_device_status",
            "pagedattn_debug_plan_dump", "pagedattn_debug_gather", "pagedattn_version",
            "pagedattn_run_decode_noalloc", "pagedattn_noalloc_device_status", "pagedattn_plan_cascade",
            "pagedattn_workspace_size_cascade")


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"pagedattn {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("force_prefill", ctypes.c_int32),
                ("decode_chunk_pages", ctypes.c_int32), ("prefill_chunk_tiles", ctypes.c_int32),
                ("force_cp_async", ctypes.c_int32), ("decode_cuda_cores", ctypes.c_int32),
                ("kv_layout", ctypes.c_int32), ("prefill_q_tiles", ctypes.c_int32),
                ("wait_limit_cycles", ctypes.c_int32), ("reserved", ctypes.c_int32 * 1)]


_I32P = ctypes.POINTER(ctypes.c_int32)
_lib = None
_lock = threading.Lock()


class PrefixGroups(ctypes.Structure):
    """pagedattn_prefix_groups: requests [group_indptr[g], group_indptr[g+1])
    share the full prefix pages prefix_page_indices[prefix_page_indptr[g] ..
    prefix_page_indptr[g+1]) ahead of their own pages."""
    _fields_ = [("group_indptr", ctypes.POINTER(ctypes.c_int32)),
                ("prefix_page_indptr", ctypes.POINTER(ctypes.c_int32)),
                ("prefix_page_indices", ctypes.POINTER(ctypes.c_int32)),
                ("num_groups", ctypes.c_int32)]


def _prefix_groups(prefix_groups):
    """(group_indptr, prefix_page_indptr, prefix_page_indices) -> (struct, arrays kept alive)."""
    arrs = [_i32(x) for x in prefix_groups]
    g = PrefixGroups()
    g.group_indptr, g.prefix_page_indptr, g.prefix_page_indices = (_ptr(a) for a in arrs)
    g.num_groups = len(arrs[0]) - 1
    return g, arrs


def load() -> ctypes.CDLL:
    """Load the shared library (built by ``attention_paged_kv_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'` "
                              "(or python -m attention_paged_kv_gb300.build); there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        plan_args = [_I32P, _I32P, _I32P, _I32P] + [ctypes.c_int32] * 6 + [ctypes.c_int, ctypes.c_int32]
        lib.pagedattn_plan.argtypes = plan_args + [ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(Options),
                                                   ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
        lib.pagedattn_plan.restype = ctypes.c_int
        lib.pagedattn_workspace_size.argtypes = plan_args + [ctypes.POINTER(Options), ctypes.POINTER(ctypes.c_size_t)]
        lib.pagedattn_workspace_size.restype = ctypes.c_int
        pg = [ctypes.POINTER(PrefixGroups)]
        lib.pagedattn_plan_cascade.argtypes = pg + lib.pagedattn_plan.argtypes
        lib.pagedattn_plan_cascade.restype = ctypes.c_int
        lib.pagedattn_workspace_size_cascade.argtypes = pg + lib.pagedattn_workspace_size.argtypes
        lib.pagedattn_workspace_size_cascade.restype = ctypes.c_int
        lib.pagedattn_run.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_void_p, ctypes.c_void_p]
        lib.pagedattn_run.restype = ctypes.c_int
        lib.pagedattn_run_stages.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_uint32]
        lib.pagedattn_run_stages.restype = ctypes.c_int
        lib.pagedattn_plan_destroy.argtypes = [ctypes.c_void_p]
        lib.pagedattn_plan_destroy.restype = ctypes.c_int
        lib.pagedattn_last_error.argtypes = []
        lib.pagedattn_last_error.restype = ctypes.c_char_p
        lib.pagedattn_device_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, _I32P]
        lib.pagedattn_device_status.restype = ctypes.c_int
        lib.pagedattn_debug_plan_dump.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_size_t)]
        lib.pagedattn_debug_plan_dump.restype = ctypes.c_int
        lib.pagedattn_debug_gather.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.pagedattn_debug_gather.restype = ctypes.c_int
        lib.pagedattn_run_decode_noalloc.argtypes = [ctypes.c_void_p] * 6
        lib.pagedattn_run_decode_noalloc.restype = ctypes.c_int
        lib.pagedattn_noalloc_device_status.argtypes = [ctypes.c_void_p, _I32P]
        lib.pagedattn_noalloc_device_status.restype = ctypes.c_int
        lib.pagedattn_version.argtypes = []
        lib.pagedattn_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def last_error() -> str:
    return load().pagedattn_last_error().decode()


def check(status: int) -> None:
    if status != PA_OK:
        raise PagedAttnError(status, last_error())


def _i32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


def dtype_code(dtype) -> int:
    import torch
    if dtype in (torch.float16, "fp16", "float16", PA_FP16):
        return PA_FP16
    if dtype in (torch.bfloat16, "bf16", "bfloat16", PA_BF16):
        return PA_BF16
    raise PagedAttnError(PA_ERR_UNSUPPORTED, f"dtype {dtype}")


PA_LAYOUT_NHD = 0
PA_LAYOUT_HND = 1


def layout_code(layout) -> int:
    """"NHD" / "HND" (or the PA_LAYOUT_* codes) -> code."""
    if layout in ("NHD", "nhd", PA_LAYOUT_NHD):
        return PA_LAYOUT_NHD
    if layout in ("HND", "hnd", PA_LAYOUT_HND):
        return PA_LAYOUT_HND
    raise PagedAttnError(PA_ERR_UNSUPPORTED, f"kv_layout {layout!r}")


def _options(num_sms=0, force_prefill=False, decode_chunk_pages=0, prefill_chunk_tiles=0,
             force_cp_async=False, decode_cuda_cores=False, kv_layout="NHD", prefill_q_tiles=0,
             wait_limit_cycles=0) -> Options:
    o = Options()
    o.num_sms = int(num_sms)
    o.force_prefill = int(bool(force_prefill))
    o.decode_chunk_pages = int(decode_chunk_pages)
    o.prefill_chunk_tiles = int(prefill_chunk_tiles)
    o.force_cp_async = int(bool(force_cp_async))
    o.decode_cuda_cores = int(bool(decode_cuda_cores))
    o.kv_layout = layout_code(kv_layout)
    o.prefill_q_tiles = int(prefill_q_tiles)
    o.wait_limit_cycles = int(wait_limit_cycles)
    return o


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def workspace_size(qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, num_qo_heads, num_kv_heads,
                   head_dim, page_size, num_pages, dtype, causal=True, prefix_groups=None, **opts) -> int:
    lib = load()
    a = [_i32(x) for x in (qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len)]
    n = ctypes.c_size_t(0)
    o = _options(**opts)
    g, _keep = _prefix_groups(prefix_groups) if prefix_groups is not None else (None, None)
    check(lib.pagedattn_workspace_size_cascade(ctypes.byref(g) if g is not None else None,
                                               _ptr(a[0]), _ptr(a[1]), _ptr(a[2]), _ptr(a[3]), len(a[0]) - 1,
                                               int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size),
                                               int(num_pages), dtype_code(dtype), int(bool(causal)), ctypes.byref(o),
                                               ctypes.byref(n)))
    return int(n.value)


class Plan:
    """A planned batch: ``begin_forward`` of the timing script.

    ``run(q, kv_cache)`` is its ``forward``; ``close()`` (or garbage
    collection) its ``end_forward``.  ``workspace``: a CUDA uint8 tensor; by
    default the plan allocates max(128 MiB, required) bytes.  ``host_only``
    builds the metadata without a device (inspection and tests).
    """

    def __init__(self, qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len, num_qo_heads, num_kv_heads,
                 head_dim, page_size, num_pages, dtype, causal=True, workspace=None, stream=None,
                 host_only=False, prefix_groups=None, **opts):
        self._lib = load()
        self._h = ctypes.c_void_p(0)
        self.num_qo_heads, self.num_kv_heads = int(num_qo_heads), int(num_kv_heads)
        self.head_dim, self.page_size, self.num_pages = int(head_dim), int(page_size), int(num_pages)
        self.dtype_code = dtype_code(dtype)
        self.kv_layout = layout_code(opts.get("kv_layout", "NHD"))
        self.causal = bool(causal)
        arrs = [_i32(x) for x in (qo_indptr, kv_page_indptr, kv_page_indices, kv_last_page_len)]
        if len(arrs[0]) < 1:
            raise PagedAttnError(PA_ERR_INVALID_ARG, "qo_indptr needs at least one entry")
        self.batch_size = len(arrs[0]) - 1
        self.total_qo = int(arrs[0][-1])
        self._arrs = arrs
        o = _options(**opts)
        ws_ptr, ws_bytes, st = None, 0, None
        if not host_only:
            import torch
            if workspace is None:
                need = workspace_size(*arrs, num_qo_heads, num_kv_heads, head_dim, page_size, num_pages, dtype,
                                      causal, prefix_groups=prefix_groups, **opts)
                workspace = torch.empty(max(need, DEFAULT_WORKSPACE_BYTES), dtype=torch.uint8, device="cuda")
            self.workspace = workspace
            ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
            st = _stream_handle(stream)
        else:
            self.workspace = None
        g, _keep = _prefix_groups(prefix_groups) if prefix_groups is not None else (None, None)
        check(self._lib.pagedattn_plan_cascade(ctypes.byref(g) if g is not None else None,
                                               _ptr(arrs[0]), _ptr(arrs[1]), _ptr(arrs[2]), _ptr(arrs[3]),
                                               self.batch_size, self.num_qo_heads, self.num_kv_heads, self.head_dim,
                                               self.page_size, self.num_pages, self.dtype_code, int(self.causal),
                                               ws_ptr, ws_bytes, ctypes.byref(o), st, ctypes.byref(self._h)))

    # -- forward
    def run(self, q, kv_cache, out=None, lse=None, stream=None, return_lse=True,
            stages: int = PA_STAGE_ALL) -> Tuple["object", Optional["object"]]:
        import torch
        T, Hq, D = self.total_qo, self.num_qo_heads, self.head_dim
        if out is None:
            out = torch.empty((T, Hq, D), dtype=q.dtype, device=q.device)
        if lse is None and return_lse:
            lse = torch.empty((T, Hq), dtype=torch.float32, device=q.device)
        for name, t in (("q", q), ("kv_cache", kv_cache), ("out", out)):
            if not t.is_cuda or not t.is_contiguous():
                raise PagedAttnError(PA_ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor")
            if dtype_code(t.dtype) != self.dtype_code:
                raise PagedAttnError(PA_ERR_INVALID_ARG, f"{name} dtype differs from the plan's")
        if tuple(q.shape) != (T, Hq, D) or tuple(out.shape) != (T, Hq, D):
            raise PagedAttnError(PA_ERR_INVALID_ARG, f"q/out must be [{T}, {Hq}, {D}]")
        want_kv = ((self.num_pages, 2, self.num_kv_heads, self.page_size, D) if self.kv_layout == PA_LAYOUT_HND
                   else (self.num_pages, 2, self.page_size, self.num_kv_heads, D))
        if tuple(kv_cache.shape) != want_kv:
            raise PagedAttnError(PA_ERR_INVALID_ARG, f"kv_cache must be {list(want_kv)}")
        if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (T, Hq) or not lse.is_contiguous()):
            raise PagedAttnError(PA_ERR_INVALID_ARG, "lse must be contiguous float32 [T, Hq]")
        check(self._lib.pagedattn_run_stages(self._h, q.data_ptr(), kv_cache.data_ptr(), out.data_ptr(),
                                             lse.data_ptr() if lse is not None else None,
                                             _stream_handle(stream), int(stages)))
        return out, lse

    forward = run

    def run_ptrs(self, q_ptr: int, kv_ptr: int, out_ptr: int, lse_ptr: Optional[int], stream: int,
                 stages: int = PA_STAGE_ALL) -> None:
        """Raw-pointer form of run (no checks beyond the library's own)."""
        check(self._lib.pagedattn_run_stages(self._h, q_ptr, kv_ptr, out_ptr, lse_ptr, stream, int(stages)))

    # -- inspection
    def dump(self) -> np.ndarray:
        n = ctypes.c_size_t(0)
        check(self._lib.pagedattn_debug_plan_dump(self._h, None, ctypes.byref(n)))
        buf = np.zeros(n.value // 4, np.int32)
        check(self._lib.pagedattn_debug_plan_dump(self._h, buf.ctypes.data_as(ctypes.c_void_p), ctypes.byref(n)))
        return buf

    def debug_gather(self, stream=None):
        import torch
        hdr = self.dump()
        off_req, B = int(hdr[21]), int(hdr[2])
        req = hdr[off_req // 4: off_req // 4 + 4 * B].reshape(-1, 4)
        kv_total = int(req[:, 2].sum()) if B else 0
        pages = torch.full((max(kv_total, 1),), -1, dtype=torch.int32, device="cuda")
        slots = torch.full((max(kv_total, 1),), -1, dtype=torch.int32, device="cuda")
        check(self._lib.pagedattn_debug_gather(self._h, pages.data_ptr(), slots.data_ptr(), _stream_handle(stream)))
        return pages[:kv_total], slots[:kv_total]

    def device_status(self, stream=None) -> int:
        flags = ctypes.c_int32(0)
        st = self._lib.pagedattn_device_status(self._h, _stream_handle(stream), ctypes.byref(flags))
        if st not in (PA_OK, PA_ERR_TIMEOUT, PA_ERR_DEVICE_CHECK):
            check(st)
        return int(flags.value)

    def close(self) -> None:
        if getattr(self, "_h", None) and self._h.value:
            self._lib.pagedattn_plan_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    end_forward = close

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def version() -> str:
    return load().pagedattn_version().decode()
