"""Python binding of libpkd.so: argument marshalling only.

Every call here checks shapes, takes raw device addresses from torch tensors
and calls the C ABI declared in ``include/pkd.h``; all arithmetic of the decode
path runs in the library's sm_103a kernels.  If the library is not built the
first call raises (there is no fallback).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkd.so")

F16, BF16, E4M3, F32 = 0, 1, 2, 3
_DTYPE_CODE = {torch.float16: F16, torch.bfloat16: BF16, torch.float8_e4m3fn: E4M3, torch.float32: F32}

DEVERR_PAGE_INDEX = 1
DEVERR_WAIT_TIMEOUT = 2


class PkdError(RuntimeError):
    """A libpkd call returned a status other than PKD_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"pkd status {status}: {message}")
        self.status = status


_lib = None

_vp = ctypes.c_void_p
# int32 host arrays are passed as plain addresses (an int per call is cheaper
# to marshal than a ctypes pointer object)
_i32p = _vp


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m paged_kv_decode_28_gb300._build` "
            "or __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    i, i64, f, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "pkd_version": (ctypes.c_char_p, []),
        "pkd_status_string": (ctypes.c_char_p, [i]),
        "pkd_last_error": (ctypes.c_char_p, []),
        "pkd_num_ctas": (i, [i, ctypes.POINTER(ctypes.c_int)]),
        "pkd_workspace_bytes": (sz, [i, i, i, i, i, i]),
        "pkd_plan_create": (i, [ctypes.POINTER(_vp), i, i, i, i, i, i, _vp, sz]),
        "pkd_plan_destroy": (i, [_vp]),
        "pkd_plan": (i, [_vp, _i32p, _vp, _i32p, i, i, i, i, i, i, i, _vp]),
        "pkd_run": (i, [_vp, _vp, _vp, _vp, i64, i64, _vp, _vp, f, _vp, _vp, _vp]),
        "pkd_cascade_decode": (i, [_vp, _vp, i, i, _vp, _vp, _vp, i64, i64, _vp, _vp, f, _vp, _vp, _vp]),
        "pkd_single_decode": (i, [_vp, _vp, _vp, i, i, i, i, i, i, _vp, _vp, f, _vp, _vp, _vp, sz, _vp]),
        "pkd_merge_state": (i, [_vp, _vp, _vp, _vp, _vp, _vp, i64, i, i, i, _vp]),
        "pkd_merge_states": (i, [_vp, _vp, i64, i, i, i, i, _vp, _vp, _vp]),
        "pkd_check_device_errors": (i, [_vp, ctypes.POINTER(ctypes.c_uint32), _vp]),
        "pkd_plan_set_timing_events": (i, [_vp, _vp, _vp]),
        "pkd_plan_set_debug": (i, [_vp, i]),
        "pkd_plan_set_kv_layout": (i, [_vp, i]),
        "pkd_mla_workspace_bytes": (sz, [i, i, i]),
        "pkd_mla_decode": (i, [_vp, _vp, _vp, _vp, _i32p, _vp, _i32p, i, i, i, i64, i64, i64, f, _vp, _vp, _vp, sz,
                               i, _vp]),
        "pkd_plan_tree": (i, [_vp, i, _vp, _vp, _vp, _vp, _i32p, _vp]),
        "pkd_tree_decode": (i, [_vp, _vp, _vp, _vp, i64, i64, f, _vp, _vp, _vp]),
        "pkd_plan_prefill": (i, [_vp, _i32p, _i32p, _vp, _i32p, i, i, i, i, i, i, i, i, _vp]),
        "pkd_prefill_run": (i, [_vp, _vp, _vp, _vp, i64, i64, f, _vp, _vp, _vp]),
        "pkd_append_kv": (i, [_vp, _vp, i, _vp, _vp, i, _vp, _vp, i, i, i, i, _vp, _vp, i, i, i64, i64, _vp, _vp,
                              _vp, _vp]),
        "pkd_decode_noalloc": (i, [_i32p, _vp, _i32p, i, i, i, i, i, i, i, i, _vp, _vp, _vp, i64, i64, _vp, _vp, f,
                                   _vp, _vp, _vp]),
        "pkd_noalloc_device_errors": (i, [ctypes.POINTER(ctypes.c_uint32), _vp]),
        "pkd_plan_host": (i, [_i32p, _i32p, i, i, i, i, _i32p, i, _i32p, _i32p, _i32p, _i32p, _i32p]),
        "pkd_prefill_units_host": (i, [_i32p, _i32p, _i32p, i, i, i, i, i, _i32p, i, ctypes.POINTER(ctypes.c_int)]),
        "pkd_tree_units_host": (i, [i, _vp, _vp, _vp, _i32p, i, i, i, i, i, i, _i32p, i,
                                    ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
        "pkd_mla_units_host": (i, [_i32p, _i32p, i, i, i, _i32p, i, ctypes.POINTER(ctypes.c_int), _i32p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int):
    if status != 0:
        raise PkdError(status, lib().pkd_last_error().decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    """The CUDA stream handle: the given torch stream's, or the current one."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _host_i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _as_i32p(a: np.ndarray) -> int:
    return a.ctypes.data


def version() -> str:
    return lib().pkd_version().decode()


_num_ctas = {}  # per device: the SM count times the decode kernel's CTAs per SM, fixed for a device


def num_ctas(device: Optional[int] = None) -> int:
    dev = torch.cuda.current_device() if device is None else int(device)
    n = _num_ctas.get(dev)
    if n is None:
        out = ctypes.c_int(0)
        _check(lib().pkd_num_ctas(dev, ctypes.byref(out)))
        n = _num_ctas[dev] = out.value
    return n


def workspace_bytes(max_batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int = 128,
                    num_ctas_: Optional[int] = None, max_prefix_splits: int = 0) -> int:
    G = num_ctas() if num_ctas_ is None else num_ctas_
    n = lib().pkd_workspace_bytes(max_batch, num_qo_heads, num_kv_heads, head_dim, G, max_prefix_splits)
    if n == 0:
        raise PkdError(1, "invalid workspace limits")
    return int(n)


# fields of one work unit, as pkd_prefill_units_host / pkd_tree_units_host return them
UNIT_FIELDS = ("q0", "q_end", "page_begin", "kv_len", "t0", "t1", "piece", "level", "diag")


def _units_call(fn, n_hint: int) -> np.ndarray:
    """Call a unit-list export with room for n_hint units, retrying once with
    the size it reports when that is too small."""
    n = ctypes.c_int(0)
    for cap in (max(n_hint, 1), None):
        cap = cap if cap is not None else max(n.value, 1)
        buf = np.zeros(cap * 12, np.int32)
        status = fn(buf, cap, n)
        if status == 0:
            return buf[: 12 * n.value].reshape(n.value, 12)[:, :9].copy()
        if status != 4 or n.value <= cap:  # not a capacity shortfall
            _check(status)
    _check(status)


def prefill_units(qo_indptr, kv_indptr, kv_last_page_len, num_qo_heads: int, num_kv_heads: int, page_size: int,
                  causal: bool = True) -> np.ndarray:
    """The work list pkd_plan_prefill uploads, built on the host (no GPU):
    int32 [n_units, 9] with the columns of UNIT_FIELDS; units 2j and 2j + 1
    are one CTA's pair."""
    qi, ki, la = _host_i32(qo_indptr), _host_i32(kv_indptr), _host_i32(kv_last_page_len)
    B = len(qi) - 1
    la_arg = la if len(la) else np.zeros(1, np.int32)
    return _units_call(lambda buf, cap, n: lib().pkd_prefill_units_host(
        _as_i32p(qi), _as_i32p(ki), _as_i32p(la_arg), B, num_qo_heads, num_kv_heads, page_size, int(bool(causal)),
        _as_i32p(buf), cap, ctypes.byref(n)), 2 * (int(qi[-1]) + B + 1))


def tree_units(levels, batch: int, num_qo_heads: int, num_kv_heads: int, page_size: int, num_ctas_: int,
               max_prefix_splits: int):
    """The work list pkd_plan_tree uploads, built on the host (no GPU), and the
    number of pieces per request row.  ``levels`` as for Plan.plan_tree but
    without the page indices: ``(req_indptr, kv_indptr, kv_last_page_len)``."""
    L = len(levels)
    ri, ki, lp = (ctypes.c_void_p * max(L, 1))(), (ctypes.c_void_p * max(L, 1))(), (ctypes.c_void_p * max(L, 1))()
    nn = np.zeros(max(L, 1), np.int32)
    keep = []
    for l, (req_indptr, kv_indptr, last) in enumerate(levels):
        r, k, la = _host_i32(req_indptr), _host_i32(kv_indptr), _host_i32(last)
        if len(la) == 0:
            la = np.zeros(1, np.int32)
        keep += [r, k, la]
        nn[l] = len(r) - 1
        ri[l], ki[l], lp[l] = r.ctypes.data, k.ctypes.data, la.ctypes.data
    pieces = ctypes.c_int(0)
    hint = 2 * max_prefix_splits * (batch + int(nn[:L].sum()) + 1)
    units = _units_call(lambda buf, cap, n: lib().pkd_tree_units_host(
        L, ri, ki, lp, _as_i32p(nn), batch, num_qo_heads, num_kv_heads, page_size, num_ctas_, max_prefix_splits,
        _as_i32p(buf), cap, ctypes.byref(n), ctypes.byref(pieces)), hint)
    del keep
    return units, int(pieces.value)


def mla_units(kv_indptr, kv_last_page_len, page_size: int, num_sms: int):
    """The key-range split of mla_decode, built on the host (no GPU): units
    int32 [n_units, 9] (UNIT_FIELDS; t0/t1 in 32-key tiles, level = output
    half) and the cut requests' piece ranges int32 [batch + 1]."""
    ki, la = _host_i32(kv_indptr), _host_i32(kv_last_page_len)
    B = len(ki) - 1
    la_arg = la if len(la) else np.zeros(1, np.int32)
    rpb = np.zeros(B + 1, np.int32)
    units = _units_call(lambda buf, cap, n: lib().pkd_mla_units_host(
        _as_i32p(ki), _as_i32p(la_arg), B, page_size, num_sms, _as_i32p(buf), cap, ctypes.byref(n),
        _as_i32p(rpb)), 2 * (B + num_sms))
    return units, rpb


def plan_host(kv_indptr, kv_last_page_len, num_kv_heads: int, page_size: int, num_ctas_: int) -> dict:
    """The library's split-KV rule evaluated on the host (no GPU needed)."""
    indptr = _host_i32(kv_indptr)
    last = _host_i32(kv_last_page_len)
    B = len(indptr) - 1
    rows = max(B * num_kv_heads, 1)
    max_items = B * num_kv_heads + num_ctas_
    items = np.zeros(max(max_items, 1) * 4, np.int32)
    cta = np.zeros(num_ctas_ + 1, np.int32)
    rb = np.zeros(rows, np.int32)
    rc = np.zeros(rows, np.int32)
    mr = np.zeros(rows, np.int32)
    counts = np.zeros(4, np.int32)
    last_arg = last if len(last) else np.zeros(1, np.int32)
    _check(lib().pkd_plan_host(_as_i32p(indptr), _as_i32p(last_arg), B, num_kv_heads, page_size, num_ctas_,
                               _as_i32p(items), max_items, _as_i32p(cta), _as_i32p(rb), _as_i32p(rc),
                               _as_i32p(mr), _as_i32p(counts)))
    n, nm = int(counts[0]), int(counts[1])
    return {
        "items": items[: 4 * n].reshape(n, 4).copy(),
        "cta_item_begin": cta.copy(),
        "row_item_begin": rb[: B * num_kv_heads].copy(),
        "row_item_count": rc[: B * num_kv_heads].copy(),
        "merge_rows": mr[:nm].copy(),
        "chunk_keys": int(counts[2]),
        "quota": int(counts[3]),
    }


# page layouts of a pool: NHD pages [page_size, Hk, D], HND pages [Hk, page_size, D]
_LAYOUT_CODE = {"NHD": 0, "HND": 1}


def _check_pool(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, kv_layout: str = "NHD"):
    """Pool geometry (N, P, Hk, D, page stride): NHD pools are
    ``[num_pages, page_size, Hk, D]``, HND pools ``[num_pages, Hk, page_size, D]``,
    each page one contiguous block."""
    if kv_layout not in _LAYOUT_CODE:
        raise ValueError("kv_layout must be 'NHD' or 'HND'")
    hnd = kv_layout == "HND"
    if k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("caches must be [num_pages, num_kv_heads, page_size, head_dim]" if hnd else
                         "caches must be [num_pages, page_size, num_kv_heads, head_dim]")
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have one shape and dtype")
    if hnd:
        N, Hk, P, D = k_cache.shape
    else:
        N, P, Hk, D = k_cache.shape
    inner = P if hnd else Hk
    for c in (k_cache, v_cache):
        # the stride of a dimension of extent 1 is never stepped (torch leaves it arbitrary)
        want = ((3, 1), (2, D), (1, inner * D))
        if any(c.shape[d] > 1 and c.stride(d) != s for d, s in want):
            raise ValueError(f"each page of the cache must be a contiguous {kv_layout} block")
    if N > 1 and k_cache.stride(0) != v_cache.stride(0):
        raise ValueError("k_cache and v_cache must share one page stride")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    return N, P, Hk, D, (k_cache.stride(0) if N > 1 else P * Hk * D)


class Plan:
    """A plan object with its device workspace: ``plan(...)`` then ``run(...)``.

    Mirrors the batch-decode wrapper of the pages: ``plan`` takes the CSR page
    table and the static geometry (host work, before CUDA-graph capture);
    ``run`` takes q and the paged K/V and returns ``(out, lse)``.
    """

    def __init__(self, max_batch: int, num_qo_heads: int, num_kv_heads: int, head_dim: int = 128,
                 max_prefix_splits: int = 0, device=None, num_ctas_: Optional[int] = None,
                 kv_layout: str = "NHD"):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(self.device):
            self.num_ctas = num_ctas() if num_ctas_ is None else int(num_ctas_)
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.max_batch = max_batch
        nbytes = workspace_bytes(max_batch, num_qo_heads, num_kv_heads, head_dim, self.num_ctas, max_prefix_splits)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        h = ctypes.c_void_p()
        _check(lib().pkd_plan_create(ctypes.byref(h), max_batch, num_qo_heads, num_kv_heads, head_dim,
                                     self.num_ctas, max_prefix_splits, _ptr(self.workspace), nbytes))
        self._h = h
        if kv_layout not in _LAYOUT_CODE:
            raise ValueError("kv_layout must be 'NHD' or 'HND'")
        self.kv_layout = kv_layout
        _check(lib().pkd_plan_set_kv_layout(h, _LAYOUT_CODE[kv_layout]))
        self._indices = None
        self.batch = 0
        self.q_dtype = self.kv_dtype = None

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.pkd_plan_destroy(h)
            self._h = None

    def plan(self, kv_indptr, kv_page_indices: torch.Tensor, kv_last_page_len, page_size: int,
             q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, stream=None):
        indptr = _host_i32(kv_indptr)
        last = _host_i32(kv_last_page_len)
        B = len(indptr) - 1
        if kv_page_indices.dtype != torch.int32 or kv_page_indices.device.type != "cuda":
            raise ValueError("kv_page_indices must be an int32 CUDA tensor")
        last_arg = last if len(last) else np.zeros(1, np.int32)
        _check(lib().pkd_plan(self._h, _as_i32p(indptr), _ptr(kv_page_indices), _as_i32p(last_arg), B,
                              self.num_qo_heads, self.num_kv_heads, self.head_dim, page_size,
                              _DTYPE_CODE[q_dtype], _DTYPE_CODE[kv_dtype], _stream(stream)))
        self._indices = kv_page_indices  # borrowed by the library until the next plan
        self.batch, self.page_size = B, page_size
        self.q_dtype, self.kv_dtype = q_dtype, kv_dtype

    def _check_geometry(self, P, Hk, D):
        if Hk != self.num_kv_heads or D != self.head_dim or (self.q_dtype is not None and P != self.page_size):
            raise ValueError(f"pool geometry (page_size {P}, kv heads {Hk}, head_dim {D}) does not match the plan "
                             f"({self.kv_layout} pages)")

    def _outputs(self, q, out, lse, B):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, self.num_qo_heads), dtype=torch.float32, device=q.device)
        return out, lse

    def run(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
            sm_scale: Optional[float] = None, k_scale: Optional[torch.Tensor] = None,
            v_scale: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        N, P, Hk, D, stride = _check_pool(q, k_cache, v_cache, self.kv_layout)
        self._check_geometry(P, Hk, D)
        if self.q_dtype is not None and q.shape != (self.batch, self.num_qo_heads, self.head_dim):
            raise ValueError(f"q must be [{self.batch}, {self.num_qo_heads}, {self.head_dim}]")
        out, lse = self._outputs(q, out, lse, q.shape[0])
        _check(lib().pkd_run(self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache), N, stride, _ptr(k_scale),
                             _ptr(v_scale), float(sm_scale or 0.0), _ptr(out), _ptr(lse), _stream(stream)))
        return out, lse

    def cascade_decode(self, prefix_page_indices: torch.Tensor, prefix_last_page_len: int, q: torch.Tensor,
                       k_cache: torch.Tensor, v_cache: torch.Tensor, *, sm_scale: Optional[float] = None,
                       k_scale=None, v_scale=None, out=None, lse=None, stream=None):
        N, P, Hk, D, stride = _check_pool(q, k_cache, v_cache, self.kv_layout)
        self._check_geometry(P, Hk, D)
        if prefix_page_indices.dtype != torch.int32 or prefix_page_indices.device.type != "cuda":
            raise ValueError("prefix_page_indices must be an int32 CUDA tensor")
        out, lse = self._outputs(q, out, lse, self.batch)
        _check(lib().pkd_cascade_decode(self._h, _ptr(prefix_page_indices), int(prefix_page_indices.numel()),
                                        int(prefix_last_page_len), _ptr(q), _ptr(k_cache), _ptr(v_cache), N,
                                        stride, _ptr(k_scale), _ptr(v_scale), float(sm_scale or 0.0),
                                        _ptr(out), _ptr(lse), _stream(stream)))
        return out, lse

    def plan_tree(self, levels, stream=None):
        """Shared levels of a prefix tree, outermost first, after ``plan`` (which
        gave each request's own pages).  Each level is ``(req_indptr, kv_indptr,
        kv_page_indices, kv_last_page_len)`` over its nodes: node n serves
        requests ``req_indptr[n] .. req_indptr[n+1]-1`` (the nodes cover the
        batch in order) and owns pages ``kv_page_indices[kv_indptr[n] ..]``
        (an int32 CUDA tensor; the others are host arrays)."""
        L = len(levels)
        if not 1 <= L <= 4:
            raise ValueError("1 to 4 shared levels")
        keep = []
        ri, ki, pi, lp = (ctypes.c_void_p * L)(), (ctypes.c_void_p * L)(), (ctypes.c_void_p * L)(), \
            (ctypes.c_void_p * L)()
        nn = np.zeros(L, np.int32)
        for l, (req_indptr, kv_indptr, idx, last) in enumerate(levels):
            r = _host_i32(req_indptr)
            k = _host_i32(kv_indptr)
            la = _host_i32(last)
            if len(la) == 0:
                la = np.zeros(1, np.int32)
            if idx.dtype != torch.int32 or idx.device.type != "cuda" or not idx.is_contiguous():
                raise ValueError("each level's kv_page_indices must be a contiguous int32 CUDA tensor")
            nn[l] = len(r) - 1
            keep += [r, k, la, idx]
            ri[l] = r.ctypes.data
            ki[l] = k.ctypes.data
            lp[l] = la.ctypes.data
            pi[l] = idx.data_ptr() if idx.numel() else None
        _check(lib().pkd_plan_tree(self._h, L, ri, ki, pi, lp, _as_i32p(nn), _stream(stream)))
        self._tree = keep  # the page-index tensors are borrowed until the next plan

    def tree_decode(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                    sm_scale: Optional[float] = None, out=None, lse=None, stream=None):
        """Decode over the prefix tree of ``plan_tree`` and the requests' own pages."""
        N, P, Hk, D, stride = _check_pool(q, k_cache, v_cache, self.kv_layout)
        self._check_geometry(P, Hk, D)
        out, lse = self._outputs(q, out, lse, self.batch)
        _check(lib().pkd_tree_decode(self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache), N, stride,
                                     float(sm_scale or 0.0), _ptr(out), _ptr(lse), _stream(stream)))
        return out, lse

    def plan_prefill(self, qo_indptr, kv_indptr, kv_page_indices: torch.Tensor, kv_last_page_len, page_size: int,
                     *, causal: bool = True, q_dtype=torch.bfloat16, kv_dtype=None, stream=None):
        """Prefill / append: request r's query tokens are rows ``qo_indptr[r] ..
        qo_indptr[r+1]-1`` of q; its keys are all of its pages (its new tokens'
        keys included); ``causal`` aligns the mask to the end of the sequence."""
        qo = _host_i32(qo_indptr)
        ip = _host_i32(kv_indptr)
        last = _host_i32(kv_last_page_len)
        B = len(ip) - 1
        if len(qo) != B + 1:
            raise ValueError("qo_indptr and kv_indptr must describe the same requests")
        if kv_page_indices.dtype != torch.int32 or kv_page_indices.device.type != "cuda":
            raise ValueError("kv_page_indices must be an int32 CUDA tensor")
        kv_dtype = q_dtype if kv_dtype is None else kv_dtype
        last_arg = last if len(last) else np.zeros(1, np.int32)
        _check(lib().pkd_plan_prefill(self._h, _as_i32p(qo), _as_i32p(ip), _ptr(kv_page_indices),
                                      _as_i32p(last_arg), B, self.num_qo_heads, self.num_kv_heads, self.head_dim,
                                      page_size, _DTYPE_CODE[q_dtype], _DTYPE_CODE[kv_dtype], int(bool(causal)),
                                      _stream(stream)))
        self._pf_indices = kv_page_indices
        self.pf_tokens, self.pf_page_size = int(qo[-1]), page_size

    def prefill(self, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, *,
                sm_scale: Optional[float] = None, out=None, lse=None, stream=None):
        """q ``[T, Hq, 128]`` -> ``(out [T, Hq, 128], lse [T, Hq])`` for the last ``plan_prefill``."""
        N, P, Hk, D, stride = _check_pool(q, k_cache, v_cache, self.kv_layout)
        if Hk != self.num_kv_heads or D != self.head_dim or P != getattr(self, "pf_page_size", P):
            raise ValueError("pool geometry does not match the prefill plan")
        if q.shape != (getattr(self, "pf_tokens", q.shape[0]), self.num_qo_heads, self.head_dim):
            raise ValueError("q must be [T, num_qo_heads, head_dim] for the planned T")
        out = torch.empty_like(q) if out is None else out
        lse = torch.empty((q.shape[0], self.num_qo_heads), dtype=torch.float32, device=q.device) if lse is None \
            else lse
        _check(lib().pkd_prefill_run(self._h, _ptr(q), _ptr(k_cache), _ptr(v_cache), N, stride,
                                     float(sm_scale or 0.0), _ptr(out), _ptr(lse), _stream(stream)))
        return out, lse

    def set_timing_events(self, start: Optional[torch.cuda.Event], stop: Optional[torch.cuda.Event]):
        """Record ``start``/``stop`` around the decode kernel of later run/cascade calls (None, None: off)."""
        a = None if start is None else ctypes.c_void_p(start.cuda_event)
        b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
        _check(lib().pkd_plan_set_timing_events(self._h, a, b))

    def set_debug(self, flags: int):
        """Test hook (PKD_DEBUG_STALL_PIPELINE = 1: later runs' decode pipelines stall
        until their waits time out and flag PKD_DEVERR_WAIT_TIMEOUT); 0 turns it off."""
        _check(lib().pkd_plan_set_debug(self._h, int(flags)))

    def check_device_errors(self, stream=None) -> int:
        flags = ctypes.c_uint32(0)
        st = lib().pkd_check_device_errors(self._h, ctypes.byref(flags), _stream(stream))
        if st not in (0, 6):
            _check(st)
        return int(flags.value)


def append_kv(k_new: torch.Tensor, v_new: torch.Tensor, batch_indices: torch.Tensor, positions: torch.Tensor,
              kv_indptr: torch.Tensor, kv_page_indices: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              *, k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
              err: Optional[torch.Tensor] = None, kv_layout: str = "NHD", stream=None):
    """Write new tokens' rows into the paged cache (in place): k_new / v_new
    ``[n, Hk, 128]``; token i goes to request ``batch_indices[i]`` at position
    ``positions[i]``.  ``kv_indptr`` / ``kv_page_indices`` are int32 CUDA tensors;
    e4m3 pools quantise with ``k_scale`` / ``v_scale``.  ``err`` (int32 CUDA
    tensor of one element) collects PKD_DEVERR_PAGE_INDEX for skipped tokens.
    ``kv_layout`` is the pools' page layout ('NHD' or 'HND')."""
    N, P, Hk, D, stride = _check_pool(k_new, k_cache, v_cache, kv_layout)
    if k_new.dim() != 3 or k_new.shape != v_new.shape or k_new.shape[1:] != (Hk, D):
        raise ValueError(f"k_new / v_new must be [n, {Hk}, {D}]")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("k_new / v_new must be contiguous")
    for t, name in ((batch_indices, "batch_indices"), (positions, "positions"), (kv_indptr, "kv_indptr"),
                    (kv_page_indices, "kv_page_indices")):
        if t.dtype != torch.int32 or t.device.type != "cuda" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    n = k_new.shape[0]
    if batch_indices.numel() != n or positions.numel() != n:
        raise ValueError("one batch index and one position per new token")
    if k_new.dtype not in (torch.float16, torch.bfloat16) or k_cache.dtype not in _DTYPE_CODE:
        raise ValueError("k_new / v_new must be f16 or bf16")
    _check(lib().pkd_append_kv(_ptr(k_new), _ptr(v_new), _DTYPE_CODE[k_new.dtype], _ptr(batch_indices),
                               _ptr(positions), n, _ptr(kv_indptr), _ptr(kv_page_indices), kv_indptr.numel() - 1,
                               Hk, D, P, _ptr(k_cache), _ptr(v_cache), _DTYPE_CODE[k_cache.dtype],
                               _LAYOUT_CODE[kv_layout], N, stride,
                               _ptr(k_scale), _ptr(v_scale), _ptr(err), _stream(stream)))


def mla_decode(q_nope: torch.Tensor, q_pe: torch.Tensor, ckv_cache: torch.Tensor, kpe_cache: torch.Tensor,
               kv_indptr, kv_page_indices: torch.Tensor, kv_last_page_len, *, sm_scale: Optional[float] = None,
               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, stream=None):
    """Multi-latent attention decode: q_nope ``[B, H, 512]`` (key up-projection
    folded in), q_pe ``[B, H, 64]``, latent pool ckv ``[N, P, 512]`` and rotary
    pool kpe ``[N, P, 64]`` (bf16) -> ``(out [B, H, 512] bf16, lse [B, H])``."""
    if q_nope.dim() != 3 or q_nope.shape[2] != 512 or q_pe.shape != q_nope.shape[:2] + (64,):
        raise ValueError("q_nope [B, H, 512] and q_pe [B, H, 64] expected")
    if ckv_cache.dim() != 3 or ckv_cache.shape[2] != 512 or kpe_cache.shape[:2] != ckv_cache.shape[:2] \
            or kpe_cache.shape[2] != 64:
        raise ValueError("ckv_cache [N, P, 512] and kpe_cache [N, P, 64] expected")
    for t in (q_nope, q_pe, ckv_cache, kpe_cache):
        if t.dtype != torch.bfloat16:
            raise ValueError("MLA decode takes bf16 tensors")
    if not (q_nope.is_contiguous() and q_pe.is_contiguous()):
        raise ValueError("q_nope / q_pe must be contiguous")
    for c, w in ((ckv_cache, 512), (kpe_cache, 64)):
        if c.stride(2) != 1 or (c.shape[1] > 1 and c.stride(1) != w):
            raise ValueError("each page of a pool must be contiguous")
    if kv_page_indices.dtype != torch.int32 or kv_page_indices.device.type != "cuda":
        raise ValueError("kv_page_indices must be an int32 CUDA tensor")
    B, H, _ = q_nope.shape
    N, P, _ = ckv_cache.shape
    indptr = _host_i32(kv_indptr)
    last = _host_i32(kv_last_page_len)
    if len(indptr) != B + 1:
        raise ValueError("kv_indptr must have batch + 1 entries")
    sms = torch.cuda.get_device_properties(q_nope.device).multi_processor_count
    nbytes = lib().pkd_mla_workspace_bytes(max(B, 1), H, sms)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_nope.device)
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=q_nope.device) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q_nope.device) if lse is None else lse
    last_arg = last if len(last) else np.zeros(1, np.int32)
    ckv_stride = ckv_cache.stride(0) if N > 1 else P * 512
    kpe_stride = kpe_cache.stride(0) if N > 1 else P * 64
    _check(lib().pkd_mla_decode(_ptr(q_nope), _ptr(q_pe), _ptr(ckv_cache), _ptr(kpe_cache), _as_i32p(indptr),
                                _ptr(kv_page_indices), _as_i32p(last_arg), B, H, P, N, ckv_stride, kpe_stride,
                                float(sm_scale or 0.0), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
                                sms, _stream(stream)))
    return out, lse, workspace


_single_ws = {}  # (device, Hq, Hk, D) -> workspace bytes of a one-request plan


def single_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, sm_scale: Optional[float] = None,
                  k_scale=None, v_scale=None, workspace: Optional[torch.Tensor] = None,
                  out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    """Quickstart call: q ``[Hq, D]``, contiguous K/V ``[kv_len, Hk, D]`` -> ``(o [Hq, D], lse [Hq])``
    (into ``out`` / ``lse`` when given)."""
    if q.dim() != 2 or k.dim() != 3 or k.shape != v.shape:
        raise ValueError("q [Hq, D] and k, v [kv_len, Hk, D] expected")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    Hq, D = q.shape
    L, Hk, _ = k.shape
    key = (q.device.index, Hq, Hk, D)
    nbytes = _single_ws.get(key)
    if nbytes is None:
        nbytes = _single_ws[key] = workspace_bytes(1, Hq, Hk, D, num_ctas(q.device.index), 0)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(Hq, dtype=torch.float32, device=q.device) if lse is None else lse
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of q's shape and dtype")
    if lse.shape != (Hq,) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 tensor [Hq]")
    _check(lib().pkd_single_decode(_ptr(q), _ptr(k), _ptr(v), L, Hq, Hk, D, _DTYPE_CODE[q.dtype],
                                   _DTYPE_CODE[k.dtype], _ptr(k_scale), _ptr(v_scale), float(sm_scale or 0.0),
                                   _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out, lse


def merge_state(v_a: torch.Tensor, s_a: torch.Tensor, v_b: torch.Tensor, s_b: torch.Tensor, *,
                out: Optional[torch.Tensor] = None, s_out: Optional[torch.Tensor] = None, stream=None):
    """State over the union of two disjoint key sets: v ``[n, H, D]``, s fp32 ``[n, H]`` (natural log)."""
    if v_a.shape != v_b.shape or v_a.dim() != 3 or s_a.shape != v_a.shape[:2] or s_b.shape != s_a.shape:
        raise ValueError("v [n, H, D] and s [n, H] expected")
    for t in (v_a, v_b, s_a, s_b):
        if not t.is_contiguous():
            raise ValueError("inputs must be contiguous")
    n, H, D = v_a.shape
    out = torch.empty_like(v_a) if out is None else out
    s_out = torch.empty_like(s_a) if s_out is None else s_out
    _check(lib().pkd_merge_state(_ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b), _ptr(out), _ptr(s_out), n, H, D,
                                 _DTYPE_CODE[v_a.dtype], _stream(stream)))
    return out, s_out


def merge_states(v: torch.Tensor, s: torch.Tensor, *, stream=None):
    """Merge k states: v ``[n, k, H, D]``, s fp32 ``[n, k, H]`` -> ``([n, H, D], [n, H])``."""
    if v.dim() != 4 or s.shape != v.shape[:3]:
        raise ValueError("v [n, k, H, D] and s [n, k, H] expected")
    if not (v.is_contiguous() and s.is_contiguous()):
        raise ValueError("inputs must be contiguous")
    n, k, H, D = v.shape
    out = torch.empty((n, H, D), dtype=v.dtype, device=v.device)
    s_out = torch.empty((n, H), dtype=torch.float32, device=v.device)
    _check(lib().pkd_merge_states(_ptr(v), _ptr(s), n, k, H, D, _DTYPE_CODE[v.dtype], _ptr(out), _ptr(s_out),
                                  _stream(stream)))
    return out, s_out


def decode_noalloc(kv_indptr, kv_page_indices: torch.Tensor, kv_last_page_len, page_size: int, q: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, *,
                   sm_scale: Optional[float] = None, k_scale=None, v_scale=None, kv_layout: str = "NHD",
                   stream=None):
    """Plan + run in one call that allocates nothing on the device: the library's
    built-in scratch area replaces the workspace (see ``pkd_decode_noalloc``).
    ``out`` and ``lse`` are caller-provided; the first call on a device must
    come before any stream capture on it, and no call runs while its stream is
    being captured.  ``kv_layout``: 'NHD' or 'HND' pools."""
    N, P, Hk, D, stride = _check_pool(q, k_cache, v_cache, kv_layout)
    indptr = _host_i32(kv_indptr)
    last = _host_i32(kv_last_page_len)
    B = len(indptr) - 1
    last_arg = last if len(last) else np.zeros(1, np.int32)
    _check(lib().pkd_decode_noalloc(_as_i32p(indptr), _ptr(kv_page_indices), _as_i32p(last_arg), B, q.shape[1],
                                    Hk, D, page_size, _DTYPE_CODE[q.dtype], _DTYPE_CODE[k_cache.dtype],
                                    _LAYOUT_CODE[kv_layout], _ptr(q),
                                    _ptr(k_cache), _ptr(v_cache), N, stride, _ptr(k_scale), _ptr(v_scale),
                                    float(sm_scale or 0.0), _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def noalloc_device_errors(stream=None) -> int:
    """PKD_DEVERR_* bits the last ``decode_noalloc`` call on the current device
    recorded (after synchronising ``stream``)."""
    flags = ctypes.c_uint32(0)
    st = lib().pkd_noalloc_device_errors(ctypes.byref(flags), _stream(stream))
    if st not in (0, 6):
        _check(st)
    return int(flags.value)
