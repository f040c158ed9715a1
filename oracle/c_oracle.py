"""ctypes front end and build step of the C fp64 oracle (``pkd_oracle.c``).

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__`` (build and
smoke) and the CPU-baseline leg of ``bench.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional

import numpy as np

try:
    import torch
except Exception:  # pragma: no cover
    torch = None

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pkd_oracle.c")
LIB = os.path.join(HERE, "libpkd_oracle.so")

_DTYPE_CODES = {"f16": 0, "bf16": 1, "e4m3": 2, "f32": 3, "f64": 4}


def build(force: bool = False) -> str:
    """Compile ``pkd_oracle.c`` with gcc + OpenMP into ``libpkd_oracle.so``."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        L.pkd_oracle_paged_decode.restype = ctypes.c_int
        L.pkd_oracle_paged_decode.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p,
        ]
        L.pkd_oracle_max_threads.restype = ctypes.c_int
        for name in ("orc_decode_bf16", "orc_decode_f16"):
            getattr(L, name).restype = ctypes.c_double
            getattr(L, name).argtypes = [ctypes.c_uint16]
        L.orc_decode_e4m3.restype = ctypes.c_double
        L.orc_decode_e4m3.argtypes = [ctypes.c_uint8]
        _lib = L
    return _lib


def _raw(t):
    """(contiguous numpy view of the raw element bits, dtype code)."""
    if torch is not None and isinstance(t, torch.Tensor):
        t = t.detach().to("cpu").contiguous()
        name = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float8_e4m3fn: "e4m3",
                torch.float32: "f32", torch.float64: "f64"}[t.dtype]
        view = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[t.element_size()]
        return t.view(view).numpy(), _DTYPE_CODES[name]
    a = np.ascontiguousarray(t)
    code = {np.float16: 0, np.float32: 3, np.float64: 4}[a.dtype.type]
    return a, code


def decode_bits(dtype: str, bits: int) -> float:
    L = lib()
    return {"bf16": L.orc_decode_bf16, "f16": L.orc_decode_f16, "e4m3": L.orc_decode_e4m3}[dtype](bits)


def max_threads() -> int:
    return int(lib().pkd_oracle_max_threads())


def paged_decode(q, k_cache, v_cache, kv_indptr, kv_page_indices, kv_last_page_len, *,
                 sm_scale: Optional[float] = None, k_scale=None, v_scale=None, rows=None,
                 num_threads: int = 0, page_stride: Optional[int] = None):
    """Same contract as ``oracle.attention.paged_decode`` (float64 results), in C.

    Caches must be ``[num_pages, P, Hk, D]`` with contiguous pages (or give
    ``page_stride`` in elements for a strided pool view).
    """
    qa, qc = _raw(q)
    B, Hq, D = qa.shape
    if torch is not None and isinstance(k_cache, torch.Tensor) and page_stride is None:
        kc = k_cache.contiguous()
        vc = v_cache.contiguous()
    else:
        kc, vc = k_cache, v_cache
    ka, kvc = _raw(kc)
    va, _ = _raw(vc)
    P, Hk = int(ka.shape[1]), int(ka.shape[2])
    if page_stride is None:
        page_stride = P * Hk * D
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    idx = np.ascontiguousarray(kv_page_indices, dtype=np.int32)
    last = np.ascontiguousarray(kv_last_page_len, dtype=np.int32)
    ks = None if k_scale is None else np.ascontiguousarray(np.asarray(
        k_scale.cpu() if torch is not None and isinstance(k_scale, torch.Tensor) else k_scale,
        dtype=np.float64))
    vs = None if v_scale is None else np.ascontiguousarray(np.asarray(
        v_scale.cpu() if torch is not None and isinstance(v_scale, torch.Tensor) else v_scale,
        dtype=np.float64))
    o = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    rows_arr = None
    n_rows = 0
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int32).reshape(-1, 2))
        n_rows = rows_arr.shape[0]
    ptr = lambda a: None if a is None else a.ctypes.data
    rc = lib().pkd_oracle_paged_decode(
        ptr(qa), qc, ptr(ka), ptr(va), kvc, int(page_stride), P, B, Hq, Hk, D,
        ptr(indptr), ptr(idx), ptr(last), float(sm_scale), ptr(ks), ptr(vs),
        ptr(rows_arr), n_rows, int(num_threads), ptr(o), ptr(lse))
    if rc != 0:
        raise RuntimeError("C oracle failed")
    return o, lse
