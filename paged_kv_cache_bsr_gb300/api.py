"""Thin ctypes binding of libpkvbsr.so (include/pkv_bsr.h).

Functions keep the C names without the ``pkv_`` prefix and only marshal
arguments: tensors become raw pointers, streams become cudaStream_t handles,
and a non-OK status becomes a ``PkvError``.  Every computation happens in the
library's CUDA kernels; there is no fallback path.  If the library has not
been built, loading raises.

``Plan`` bundles a plan handle with the device workspace and the pinned host
staging buffer it needs (allocated with torch, i.e. by the caller).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

from . import build as _build

PKV_OK = 0
PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2
PLAN_DECODE, PLAN_PREFILL, PLAN_MIXED = 0, 1, 2

_DTYPES = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32}


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Params(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("page_size", ctypes.c_int), ("dtype", ctypes.c_int), ("sm_scale", ctypes.c_float),
                ("logits_cap", ctypes.c_float), ("causal", ctypes.c_int)]


class Limits(ctypes.Structure):
    _fields_ = [("max_batch", ctypes.c_int), ("max_total_q", ctypes.c_int64), ("max_kv_pages", ctypes.c_int64)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("grid_ctas", ctypes.c_int), ("workers", ctypes.c_int), ("active_workers", ctypes.c_int),
                ("num_work", ctypes.c_int), ("num_merge", ctypes.c_int), ("num_slots", ctypes.c_int),
                ("max_cost", ctypes.c_int64), ("total_cost", ctypes.c_int64),
                ("prefill_ctas", ctypes.c_int), ("decode_ctas", ctypes.c_int)]


_lib = None
_lock = threading.Lock()

EXPORTS = [
    "pkv_status_string", "pkv_version", "pkv_plan_create", "pkv_plan_create_host", "pkv_plan_destroy",
    "pkv_plan_workspace_bytes", "pkv_plan_compute", "pkv_plan_run", "pkv_plan_get_info", "pkv_plan_get_work",
    "pkv_batch_decode_paged", "pkv_batch_prefill_paged", "pkv_merge_state", "pkv_merge_states",
    "pkv_get_device_error",
    "pkv_plan_set_timing_events", "pkv_batch_decode_paged_noalloc", "pkv_append_paged_kv",
    "pkv_batch_prefill_paged_masked", "pkv_batch_mixed_paged", "pkv_plan_set_pipelined",
    "pkv_plan_set_split_kv",
]


def library_path() -> str:
    return _build.LIB_PATH


def load(path: Optional[str] = None):
    """Load libpkvbsr.so (raises if it is missing: there is no CPU path)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or library_path()
        if not os.path.exists(p):
            raise RuntimeError(f"libpkvbsr.so is not built ({p}); run paged_kv_cache_bsr_gb300.build.build()")
        lib = ctypes.CDLL(p)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "pkv_status_string": (ctypes.c_char_p, [i32]),
            "pkv_version": (i32, []),
            "pkv_plan_create": (i32, [ctypes.POINTER(vp), i32, ctypes.POINTER(Params), ctypes.POINTER(Limits), i32]),
            "pkv_plan_create_host": (i32, [ctypes.POINTER(vp), i32, ctypes.POINTER(Params), ctypes.POINTER(Limits), i32]),
            "pkv_plan_destroy": (i32, [vp]),
            "pkv_plan_workspace_bytes": (i32, [vp, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
            "pkv_plan_compute": (i32, [vp, i32, vp, vp, vp, vp, i64, vp, sz]),
            "pkv_plan_run": (i32, [vp, i32, vp, vp, vp, vp, i64, vp, sz, vp, sz, vp]),
            "pkv_plan_get_info": (i32, [vp, ctypes.POINTER(PlanInfo)]),
            "pkv_plan_get_work": (i32, [vp, vp, i64, ctypes.POINTER(i64)]),
            "pkv_batch_decode_paged": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_batch_prefill_paged": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_merge_state": (i32, [vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, vp]),
            "pkv_merge_states": (i32, [vp, vp, i32, i64, vp, vp, i64, i32, i32, i32, vp]),
            "pkv_get_device_error": (i32, [vp, vp, ctypes.POINTER(i32), i32, vp]),
            "pkv_plan_set_timing_events": (i32, [vp, vp, vp]),
            "pkv_batch_decode_paged_noalloc": (i32, [vp, vp, sz, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_batch_prefill_paged_masked": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp]),
            "pkv_batch_mixed_paged": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "pkv_plan_set_pipelined": (i32, [vp, i32]),
            "pkv_plan_set_split_kv": (i32, [vp, i32]),
            "pkv_append_paged_kv": (i32, [ctypes.POINTER(Params), i32, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp,
                                          vp, ctypes.c_double, vp, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().pkv_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def _check(st: int, what: str) -> None:
    if st != PKV_OK:
        raise PkvError(st, what)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libpkvbsr must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def dtype_code(dtype: torch.dtype) -> int:
    return _DTYPES[dtype]


def make_params(num_qo_heads, num_kv_heads, head_dim, page_size, dtype, sm_scale, logits_cap=0.0,
                causal=False) -> Params:
    return Params(int(num_qo_heads), int(num_kv_heads), int(head_dim), int(page_size),
                  dtype_code(dtype) if isinstance(dtype, torch.dtype) else int(dtype), float(sm_scale),
                  float(logits_cap), int(bool(causal)))


# ----------------------------------------------------------------------------- C names
def plan_create(kind: int, params: Params, limits: Limits, device: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load().pkv_plan_create(ctypes.byref(h), kind, ctypes.byref(params), ctypes.byref(limits), device),
           "pkv_plan_create")
    return h


def plan_create_host(kind: int, params: Params, limits: Limits, num_sms: int) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(load().pkv_plan_create_host(ctypes.byref(h), kind, ctypes.byref(params), ctypes.byref(limits),
                                       num_sms), "pkv_plan_create_host")
    return h


def plan_destroy(h) -> None:
    _check(load().pkv_plan_destroy(h), "pkv_plan_destroy")


def plan_workspace_bytes(h) -> Tuple[int, int]:
    d, hb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().pkv_plan_workspace_bytes(h, ctypes.byref(d), ctypes.byref(hb)), "pkv_plan_workspace_bytes")
    return d.value, hb.value


def _host_i32(t):
    if t is None:
        return None
    t = torch.as_tensor(t, dtype=torch.int32)
    if t.is_cuda:
        raise ValueError("plan arrays must be host tensors")
    return t.contiguous()


def plan_compute(h, batch: int, qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h, num_pages: int,
                 host_ws: torch.Tensor) -> None:
    qo, ip, ix, la = (_host_i32(x) for x in (qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h))
    _check(load().pkv_plan_compute(h, int(batch), _ptr(qo), _ptr(ip), _ptr(ix), _ptr(la), int(num_pages),
                                   _ptr(host_ws), host_ws.numel() * host_ws.element_size()), "pkv_plan_compute")


def plan_run(h, batch: int, qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h, num_pages: int,
             dev_ws: torch.Tensor, host_ws: torch.Tensor, stream=None) -> None:
    qo, ip, ix, la = (_host_i32(x) for x in (qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h))
    _check(load().pkv_plan_run(h, int(batch), _ptr(qo), _ptr(ip), _ptr(ix), _ptr(la), int(num_pages),
                               _ptr(dev_ws), dev_ws.numel() * dev_ws.element_size(), _ptr(host_ws),
                               host_ws.numel() * host_ws.element_size(), _stream(stream)), "pkv_plan_run")


def plan_set_split_kv(h, on: bool) -> None:
    """Decode plans: split-KV on (default) or off (each page list whole on one worker)."""
    _check(load().pkv_plan_set_split_kv(h, int(bool(on))), "pkv_plan_set_split_kv")


def plan_get_info(h) -> PlanInfo:
    info = PlanInfo()
    _check(load().pkv_plan_get_info(h, ctypes.byref(info)), "pkv_plan_get_info")
    return info


def plan_get_work(h) -> torch.Tensor:
    n = ctypes.c_int64()
    lib = load()
    lib.pkv_plan_get_work(h, None, 0, ctypes.byref(n))
    out = torch.empty((n.value, 8), dtype=torch.int32)
    if n.value:
        _check(lib.pkv_plan_get_work(h, _ptr(out), n.value, ctypes.byref(n)), "pkv_plan_get_work")
    return out


def batch_decode_paged(h, q, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse, dev_ws, stream=None) -> None:
    _check(load().pkv_batch_decode_paged(h, _ptr(q), _ptr(kv_data), _ptr(kv_indices), _ptr(kv_indptr),
                                         _ptr(kv_last_page_len), _ptr(o), _ptr(lse), _ptr(dev_ws),
                                         _stream(stream)), "pkv_batch_decode_paged")


def batch_decode_paged_noalloc(h, host_tables, q, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse,
                               stream=None) -> None:
    """Decode with the library's static device scratch instead of a caller workspace.

    ``host_tables`` is the host buffer ``plan_compute`` filled for this plan.
    """
    _check(load().pkv_batch_decode_paged_noalloc(h, _ptr(host_tables),
                                                 host_tables.numel() * host_tables.element_size(), _ptr(q),
                                                 _ptr(kv_data), _ptr(kv_indices), _ptr(kv_indptr),
                                                 _ptr(kv_last_page_len), _ptr(o), _ptr(lse), _stream(stream)),
           "pkv_batch_decode_paged_noalloc")


def batch_prefill_paged(h, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse, dev_ws,
                        stream=None) -> None:
    _check(load().pkv_batch_prefill_paged(h, _ptr(q), _ptr(qo_indptr), _ptr(kv_data), _ptr(kv_indices),
                                          _ptr(kv_indptr), _ptr(kv_last_page_len), _ptr(o), _ptr(lse),
                                          _ptr(dev_ws), _stream(stream)), "pkv_batch_prefill_paged")


def batch_prefill_paged_masked(h, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len, packed_mask,
                               o, lse, dev_ws, stream=None) -> None:
    """Prefill with a packed custom mask (uint8 device tensor, whole 32-bit words)."""
    _check(load().pkv_batch_prefill_paged_masked(h, _ptr(q), _ptr(qo_indptr), _ptr(kv_data), _ptr(kv_indices),
                                                 _ptr(kv_indptr), _ptr(kv_last_page_len), _ptr(packed_mask),
                                                 packed_mask.numel() * packed_mask.element_size(), _ptr(o),
                                                 _ptr(lse), _ptr(dev_ws), _stream(stream)),
           "pkv_batch_prefill_paged_masked")


def batch_mixed_paged(h, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse, dev_ws,
                      stream=None) -> None:
    _check(load().pkv_batch_mixed_paged(h, _ptr(q), _ptr(qo_indptr), _ptr(kv_data), _ptr(kv_indices),
                                        _ptr(kv_indptr), _ptr(kv_last_page_len), _ptr(o), _ptr(lse), _ptr(dev_ws),
                                        _stream(stream)), "pkv_batch_mixed_paged")


def merge_state(o_a, lse_a, o_b, lse_b, o_out, lse_out=None, stream=None) -> None:
    """merge_state over [n_rows, num_heads, head_dim] states (dtype fp16/bf16/fp32)."""
    if o_a.dim() != 3:
        raise ValueError("o must be [n_rows, num_heads, head_dim]")
    n, hh, d = o_a.shape
    _check(load().pkv_merge_state(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out), _ptr(lse_out),
                                  n, hh, d, dtype_code(o_a.dtype), _stream(stream)), "pkv_merge_state")


def merge_states(o_states, lse_states, num_states: int, o_out, lse_out=None, stream=None) -> None:
    """merge_state over ``num_states`` states laid out one after another: o_states is
    [num_states * n_rows, num_heads, head_dim] (fp16/bf16/fp32) and lse_states
    [num_states * n_rows, num_heads]; o_out [n_rows, num_heads, head_dim] may be the
    rows of one of the states."""
    if o_states.dim() != 3 or o_states.shape[0] % num_states:
        raise ValueError("o_states must be [num_states * n_rows, num_heads, head_dim]")
    rows, hh, d = o_states.shape
    n = rows // num_states
    _check(load().pkv_merge_states(_ptr(o_states), _ptr(lse_states), int(num_states), n, _ptr(o_out), _ptr(lse_out),
                                   n, hh, d, dtype_code(o_states.dtype), _stream(stream)), "pkv_merge_states")


def append_paged_kv(params: Params, append_indptr, kv_indptr, kv_indices, kv_last_page_len, k_new, v_new,
                    kv_data, q_in=None, q_out=None, rope_theta: float = 0.0, error=None, stream=None) -> None:
    """Write new tokens' K/V into their pages (page table already including them);
    with rope_theta > 0 rotate the keys and, when given, the queries (q_out may be q_in)."""
    batch = int(append_indptr.numel()) - 1
    nnz = int(k_new.shape[0])
    if q_in is not None and q_out is None:
        q_out = q_in
    _check(load().pkv_append_paged_kv(ctypes.byref(params), batch, nnz, int(kv_data.shape[0]), _ptr(append_indptr),
                                      _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(k_new),
                                      _ptr(v_new), _ptr(kv_data), _ptr(q_in), _ptr(q_out), float(rope_theta),
                                      _ptr(error), _stream(stream)), "pkv_append_paged_kv")


def plan_set_timing_events(h, start=None, stop=None) -> None:
    """Record torch.cuda.Event ``start``/``stop`` around the main kernel of later run calls."""
    def handle(ev):
        if ev is None:
            return None
        if not ev.cuda_event:
            ev.record()  # torch creates the event lazily
        return ctypes.c_void_p(ev.cuda_event)
    _check(load().pkv_plan_set_timing_events(h, handle(start), handle(stop)), "pkv_plan_set_timing_events")


def get_device_error(h, dev_ws, clear: bool = False, stream=None) -> int:
    code = ctypes.c_int()
    _check(load().pkv_get_device_error(h, _ptr(dev_ws), ctypes.byref(code), int(clear), _stream(stream)),
           "pkv_get_device_error")
    return code.value


# ----------------------------------------------------------------------------- convenience
class Plan:
    """A plan handle plus the caller-side buffers it needs.

    ``kind`` is PLAN_DECODE, PLAN_PREFILL or PLAN_MIXED.  The device workspace and the
    pinned host staging buffer are allocated once here, with torch, for the
    given limits; ``plan()`` re-plans a new batch into them and ``run()``
    launches the kernels.
    """

    def __init__(self, kind: int, *, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 dtype: torch.dtype, sm_scale: float, logits_cap: float = 0.0, causal: bool = False,
                 max_batch: int, max_total_q: Optional[int] = None, max_kv_pages: int,
                 device: Optional[int] = None, pipelined: bool = False, split_kv: bool = True):
        self.kind = kind
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.params = make_params(num_qo_heads, num_kv_heads, head_dim, page_size, dtype, sm_scale, logits_cap,
                                  causal)
        self.limits = Limits(int(max_batch), int(max_batch if max_total_q is None else max_total_q),
                             int(max_kv_pages))
        self.handle = plan_create(kind, self.params, self.limits, self.device)
        dev_bytes, host_bytes = plan_workspace_bytes(self.handle)
        self.dev_ws = torch.empty(dev_bytes, dtype=torch.uint8, device=f"cuda:{self.device}")
        self.host_ws = torch.empty(host_bytes, dtype=torch.uint8, pin_memory=True)
        self.num_pages = 0
        if pipelined:
            _check(load().pkv_plan_set_pipelined(self.handle, 1), "pkv_plan_set_pipelined")
        if not split_kv:
            plan_set_split_kv(self.handle, False)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _lib is not None:
            try:
                _lib.pkv_plan_destroy(h)
            except Exception:
                pass
            self.handle = None

    def plan(self, kv_indptr_h, kv_last_page_len_h, num_pages: int, *, qo_indptr_h=None, kv_indices_h=None,
             stream=None) -> None:
        batch = int(torch.as_tensor(kv_indptr_h).numel()) - 1
        plan_run(self.handle, batch, qo_indptr_h, kv_indptr_h, kv_indices_h, kv_last_page_len_h, num_pages,
                 self.dev_ws, self.host_ws, stream)
        self.num_pages = int(num_pages)

    def run(self, q, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse=None, *, qo_indptr=None,
            mask=None, stream=None) -> None:
        if mask is not None:
            if self.kind != PLAN_PREFILL:
                raise ValueError("a custom mask needs a prefill plan")
            batch_prefill_paged_masked(self.handle, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len,
                                       mask, o, lse, self.dev_ws, stream)
        elif self.kind == PLAN_MIXED:
            batch_mixed_paged(self.handle, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse,
                              self.dev_ws, stream)
        elif self.kind == PLAN_DECODE:
            batch_decode_paged(self.handle, q, kv_data, kv_indices, kv_indptr, kv_last_page_len, o, lse,
                               self.dev_ws, stream)
        else:
            batch_prefill_paged(self.handle, q, qo_indptr, kv_data, kv_indices, kv_indptr, kv_last_page_len, o,
                                lse, self.dev_ws, stream)

    def info(self) -> PlanInfo:
        return plan_get_info(self.handle)

    def work(self) -> torch.Tensor:
        return plan_get_work(self.handle)

    def set_timing_events(self, start=None, stop=None) -> None:
        plan_set_timing_events(self.handle, start, stop)

    def device_error(self, clear: bool = False, stream=None) -> int:
        return get_device_error(self.handle, self.dev_ws, clear, stream)
