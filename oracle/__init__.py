"""fp64 CPU oracle for paged (block-sparse row) KV-cache attention.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg are the only callers.  The
product package never imports this module, and this module never imports the
product package: it takes plain host arrays (numpy, or torch CPU tensors) and
shares no code, header or table with the CUDA path.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, OpenMP over
(query row, head) pairs); this file compiles it with gcc and marshals
arguments through ctypes.  Every function follows the FlashInfer pages:

* ``gather``        -- page-table gather ("FlashInfer" guide, section 2
                       "Page-Level Attention").
* ``attention``     -- softmax(scale * Q K^T) V over the gathered keys, with the
                       logit soft-cap transform (fdeinterviews summary,
                       "Customizable attention") and the end-aligned causal
                       mask of ``causal=True`` prefill ("The Interface").
* ``merge_states``  -- log-sum-exp composition of attention states (guide,
                       section 3, "Cascade Attention" / "FlashDecoding").
* ``cascade``       -- shared-prefix attention computed once for the whole
                       row block, per-request suffix attention, then a merge
                       (guide section 3, "Cascade Attention"; fdeinterviews
                       "One format", composable formats); any number of levels.
* ``rope``, ``append_positions``, ``append_paged_kv`` -- the append stage that
                       writes new tokens into their pages (greptalks
                       summary, Background, "Dynamic Problem Shapes") with
                       the rotary query/key transform (fdeinterviews
                       summary, "Customizable attention"), in plain numpy
                       fp64.
* ``encode16``      -- fp64 -> fp16/bf16 storage, round to nearest even.

Parity pins: see tests/test_oracle_pins.py.  Every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math).  Returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = ctypes.POINTER(ctypes.c_int32)
            i64p = ctypes.POINTER(ctypes.c_int64)
            u16p = ctypes.POINTER(ctypes.c_uint16)
            f64p = ctypes.POINTER(ctypes.c_double)
            lib.pkv_oracle_attention.restype = ctypes.c_int
            lib.pkv_oracle_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                u16p, ctypes.c_int64, i32p, u16p, ctypes.c_int64, i32p, i32p, i32p,
                ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_void_p, i64p, ctypes.c_int64,
                f64p, f64p, ctypes.c_int]
            lib.pkv_oracle_gather.restype = ctypes.c_int
            lib.pkv_oracle_gather.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                u16p, ctypes.c_int64, i32p, i32p, i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                f64p, ctypes.c_int64]
            lib.pkv_oracle_merge_states.restype = None
            lib.pkv_oracle_merge_states.argtypes = [
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, f64p, f64p, f64p, f64p]
            lib.pkv_oracle_decode16.restype = None
            lib.pkv_oracle_decode16.argtypes = [u16p, f64p, ctypes.c_int64, ctypes.c_int]
            lib.pkv_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    """Raw 16-bit storage of an fp16/bf16 array (torch CPU tensor or numpy)."""
    if hasattr(x, "detach"):  # torch tensor, viewed as raw bits without importing torch here
        x = x.detach().contiguous().view(dtype=_torch_int16()).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype.itemsize != 2:
        raise TypeError(f"expected a 16-bit storage array, got {a.dtype}")
    return a.view(np.uint16)


def _torch_int16():
    import torch  # only for viewing the caller's tensors as raw bits
    return torch.int16


def _dtype_code(x, dtype: Optional[str]) -> int:
    if dtype is not None:
        return {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16}[dtype]
    name = str(getattr(x, "dtype", ""))
    if "bfloat16" in name:
        return BF16
    if "float16" in name:
        return F16
    raise TypeError(f"cannot tell fp16 from bf16 for {name!r}; pass dtype=")


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(_load().pkv_oracle_num_threads())


def decode16(x, dtype: Optional[str] = None) -> np.ndarray:
    """Exact fp64 values of 16-bit storage (the decoding every oracle routine uses)."""
    code = _dtype_code(x, dtype)
    a = _u16(x)
    out = np.empty(a.shape, dtype=np.float64)
    _load().pkv_oracle_decode16(_ptr(a, ctypes.c_uint16), _ptr(out, ctypes.c_double), a.size, code)
    return out


def gather(kv_data, kv_indptr, kv_indices, kv_last_page_len, b: int, kv_sel: int, kvh: int,
           dtype: Optional[str] = None) -> np.ndarray:
    """Request b's K (kv_sel=0) or V (kv_sel=1) rows for kv head ``kvh``: [kv_len, head_dim]."""
    code = _dtype_code(kv_data, dtype)
    kv = _u16(kv_data)
    num_pages, _, hkv, page_size, d = kv.shape
    indptr, indices, last = _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    batch = indptr.size - 1
    n_pages = int(indptr[b + 1] - indptr[b]) if 0 <= b < batch else 0
    out = np.empty((max(n_pages * page_size, 1), d), dtype=np.float64)
    n = _load().pkv_oracle_gather(batch, hkv, d, page_size, code, _ptr(kv, ctypes.c_uint16),
                                  num_pages, _ptr(indptr, ctypes.c_int32),
                                  _ptr(indices, ctypes.c_int32), _ptr(last, ctypes.c_int32),
                                  b, kv_sel, kvh, _ptr(out, ctypes.c_double), out.shape[0])
    if n < 0:
        raise ValueError(f"oracle gather rejected the page table (status {n})")
    return out[:n]


def attention(q, kv_data, qo_indptr, kv_indptr, kv_indices, kv_last_page_len, *,
              sm_scale: float, causal: bool = False, logits_cap: float = 0.0,
              rows: Optional[Sequence[int]] = None, threads: int = 0,
              dtype: Optional[str] = None, mask=None) -> Tuple[np.ndarray, np.ndarray]:
    """fp64 attention over the paged KV cache.

    q [total_q, Hq, d], kv_data [num_pages, 2, Hkv, page_size, d] (16-bit storage).
    Returns (o [n, Hq, d], lse [n, Hq]) for the listed global rows (all rows when
    ``rows`` is None); lse is the natural log-sum-exp of the (capped) logits.
    ``mask``: packed custom-mask bytes (request b's [qo_len, kv_len] boolean matrix,
    row-major, least significant bit first, requests back to back from bit 0), or None.
    """
    code = _dtype_code(q, dtype)
    qa, kv = _u16(q), _u16(kv_data)
    total_q, hq, d = qa.shape
    num_pages, two, hkv, page_size, d2 = kv.shape
    if two != 2 or d2 != d:
        raise ValueError("kv_data must be [num_pages, 2, num_kv_heads, page_size, head_dim]")
    qo, indptr, indices, last = _i32(qo_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    batch = indptr.size - 1
    if rows is None:
        row_arr = None
        n = total_q
    else:
        row_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = row_arr.size
    mask_arr = None
    if mask is not None:
        if hasattr(mask, "detach"):
            mask = mask.detach().cpu().numpy()
        mask_arr = np.ascontiguousarray(np.asarray(mask).view(np.uint8).reshape(-1))
        kv_lens = [((int(indptr[b + 1]) - int(indptr[b])) - 1) * page_size + int(last[b])
                   if indptr[b + 1] > indptr[b] else 0 for b in range(batch)]
        bits = sum((int(qo[b + 1]) - int(qo[b])) * kv_lens[b] for b in range(batch))
        if mask_arr.size * 8 < bits:
            raise ValueError(f"mask holds {mask_arr.size * 8} bits, the batch needs {bits}")
    o = np.empty((n, hq, d), dtype=np.float64)
    lse = np.empty((n, hq), dtype=np.float64)
    st = _load().pkv_oracle_attention(
        batch, hq, hkv, d, page_size, code, _ptr(qa, ctypes.c_uint16), total_q,
        _ptr(qo, ctypes.c_int32), _ptr(kv, ctypes.c_uint16), num_pages,
        _ptr(indptr, ctypes.c_int32), _ptr(indices, ctypes.c_int32), _ptr(last, ctypes.c_int32),
        int(bool(causal)), float(sm_scale), float(logits_cap),
        None if mask_arr is None else mask_arr.ctypes.data_as(ctypes.c_void_p),
        None if row_arr is None else _ptr(row_arr, ctypes.c_int64), n,
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(threads))
    if st != 0:
        raise ValueError(f"oracle rejected the inputs (status {st})")
    return o, lse


def attention_of(batch, rows=None, threads: int = 0, mask=None):
    """``attention`` on a workload object with the fields of a paged batch."""
    return attention(batch.q, batch.kv_data, batch.qo_indptr, batch.kv_indptr, batch.kv_indices,
                     batch.kv_last_page_len, sm_scale=batch.sm_scale, causal=batch.causal,
                     logits_cap=batch.logits_cap, rows=rows, threads=threads, mask=mask)


def merge_states(os_, lses) -> Tuple[np.ndarray, np.ndarray]:
    """Merge states (o_i [..., d], lse_i [...]) over disjoint key sets (fp64)."""
    o = np.ascontiguousarray(np.stack([np.asarray(x, dtype=np.float64) for x in os_]))
    lse = np.ascontiguousarray(np.stack([np.asarray(x, dtype=np.float64) for x in lses]))
    k = o.shape[0]
    d = o.shape[-1]
    lead = o.shape[1:-1]
    if lse.shape[1:] != lead:
        raise ValueError("lse shapes must match o without its last axis")
    n = int(np.prod(lead)) if lead else 1
    o2 = o.reshape(k, n, d)
    l2 = lse.reshape(k, n)
    out = np.empty((n, d), dtype=np.float64)
    lout = np.empty((n,), dtype=np.float64)
    _load().pkv_oracle_merge_states(k, n, d, _ptr(o2, ctypes.c_double), _ptr(l2, ctypes.c_double),
                                    _ptr(out, ctypes.c_double), _ptr(lout, ctypes.c_double))
    return out.reshape(*lead, d), lout.reshape(lead)


def cascade(*level_batches, threads: int = 0):
    """Cascade (shared-prefix) attention over a prefix tree, level by level, merged.

    Two levels are the common case: a prefix batch holding every request's query as
    one row block against the shared prefix pages, and a suffix batch holding each
    request against its own pages.  More levels (a system prompt, per-group prompts,
    per-request tokens) follow the same rule: each level's batch groups the request
    rows into consecutive blocks, each block against its own pages.  All views index
    the same pool.  Returns (o, lse) per request row: the merge of the levels'
    states (greptalks summary, "Composable Formats for Shared Prefixes": one
    block-sparse matrix decomposed into several of different block sizes).
    """
    if len(level_batches) < 1:
        raise ValueError("cascade needs at least one level")
    states = [attention_of(b, threads=threads) for b in level_batches]
    return merge_states([s[0] for s in states], [s[1] for s in states])


# ----------------------------------------------------------------------------- append stage
def encode16(x, dtype: str) -> np.ndarray:
    """Round fp64 values to the nearest fp16 / bf16 value, ties to even (the IEEE
    default), returned as fp64 holding exactly representable values.

    A finite x = m * 2^e with m in [0.5, 1) has its unit in the last place at
    2^(e - bits) for a format of ``bits`` significant bits, but never below the
    format's smallest subnormal; values past the largest finite one become inf.
    """
    bits, min_exp, max_finite = {"bf16": (8, -133, 3.3895313892515355e38),
                                 "f16": (11, -24, 65504.0)}[dtype]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    _, e = np.frexp(x[fin])
    ulp_exp = np.maximum(e - bits, min_exp).astype(np.int64)
    r = np.ldexp(np.rint(np.ldexp(x[fin], -ulp_exp)), ulp_exp)
    # past the largest finite value by half an ulp or more: infinity
    top_ulp = 2.0 ** (int(np.frexp(max_finite)[1]) - bits)
    r = np.where(np.abs(x[fin]) >= max_finite + top_ulp / 2, np.copysign(np.inf, x[fin]), r)
    out[fin] = r
    return out


def rope(x, positions, theta: float, dtype: Optional[str] = None) -> np.ndarray:
    """Rotary position embedding (RoFormer), "rotate half" pairing, in fp64.

    x [n, H, d] (16-bit storage decoded exactly, or any float array); row t turns by
    positions[t]: element i < d/2 pairs with i + d/2 and the pair turns by the angle
    positions[t] * theta^(-2i/d):  (a, b) -> (a cos - b sin, b cos + a sin).
    """
    xv = _as_f64(x, dtype)
    n, _, d = xv.shape
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(positions, dtype=np.float64).reshape(n)[:, None] * inv_freq[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = xv[..., :half], xv[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _as_f64(x, dtype: Optional[str]) -> np.ndarray:
    """16-bit storage decoded exactly; any other float array as fp64."""
    name = str(getattr(x, "dtype", ""))
    if dtype is not None or "float16" in name:
        return decode16(x, dtype)
    return np.asarray(x, dtype=np.float64)


def append_positions(append_indptr, kv_indptr, kv_last_page_len, kv_indices, page_size: int):
    """Where each new token goes.  The page table already holds the new tokens, and
    request b's n_b new tokens are its last n_b: token i of them sits at position
    kv_len_b - n_b + i, in page kv_indices[kv_indptr[b] + pos // P], slot pos % P.

    Returns (request, position, page, slot), one entry per new token.
    """
    ap, ip, ix, last = _i32(append_indptr), _i32(kv_indptr), _i32(kv_indices), _i32(kv_last_page_len)
    batch = ip.size - 1
    if ap.size != batch + 1 or ap[0] != 0 or np.any(np.diff(ap) < 0):
        raise ValueError("append_indptr must start at 0 and be non-decreasing, one entry per request + 1")
    req, pos, page, slot = [], [], [], []
    for b in range(batch):
        n_pages = int(ip[b + 1] - ip[b])
        kv_len = (n_pages - 1) * page_size + int(last[b]) if n_pages > 0 else 0
        n_new = int(ap[b + 1] - ap[b])
        if n_new > kv_len:
            raise ValueError(f"request {b}: {n_new} new tokens but kv_len {kv_len}")
        for i in range(n_new):
            p = kv_len - n_new + i
            req.append(b)
            pos.append(p)
            page.append(int(ix[ip[b] + p // page_size]))
            slot.append(p % page_size)
    as64 = lambda v: np.asarray(v, dtype=np.int64)
    return as64(req), as64(pos), as64(page), as64(slot)


def append_paged_kv(kv_data, append_indptr, kv_indptr, kv_indices, kv_last_page_len, k_new, v_new,
                    rope_theta: float = 0.0):
    """The KV pool after appending new tokens, in fp64.

    kv_data [num_pages, 2, Hkv, P, d] (16-bit storage); k_new, v_new [nnz, Hkv, d].
    The keys turn by their positions when rope_theta > 0 (``rope``); values never do.
    Returns (kv fp64 with the new tokens written, page [nnz], slot [nnz]).
    """
    kv = decode16(kv_data)
    page_size = kv.shape[3]
    _, pos, page, slot = append_positions(append_indptr, kv_indptr, kv_last_page_len, kv_indices, page_size)
    if len(set(zip(page.tolist(), slot.tolist()))) != page.size:
        raise ValueError("two new tokens map to the same page slot")
    if np.any(page < 0) or np.any(page >= kv.shape[0]):
        raise ValueError("page id out of range")
    k = rope(k_new, pos, rope_theta) if rope_theta > 0 else decode16(k_new)
    v = decode16(v_new)
    kv[page, 0, :, slot, :] = k
    kv[page, 1, :, slot, :] = v
    return kv, page, slot
