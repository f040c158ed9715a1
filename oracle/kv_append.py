"""CPU oracle for appending new keys / values to a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/`` and the measurement leg of ``bench.py`` may call it.  It shares
no code with the CUDA path.

The write step around each decode step: the new token's K and V rows go into
the request's pages (README mirror, "Core Features": decode, prefill and
*append* kernels over a paged and ragged KV cache; deep dive, "The Code,
Annotated", snippet one: request b owns pages ``indices[indptr[b]:indptr[b+1]]``
in order, ``page_size`` slots each, NHD layout).  The pages name the step but
print no definition; the plainest reading, used here:

* token i of the new ones belongs to request ``batch_indices[i]`` at position
  ``positions[i]`` of its sequence; its rows go to page
  ``indices[indptr[b] + pos // page_size]``, slot ``pos % page_size``, every kv
  head, and nothing else of the cache changes;
* a 16-bit pool stores the new values unchanged;
* an e4m3 pool stores ``e4m3(x / scale[h])`` with the quotient taken in float32
  (the precision the kernel takes it in, since the code is an integer decided
  by floating point), rounded to the nearest E4M3 value with ties to even, and
  saturated to +-448 (the largest finite E4M3 value) instead of overflowing;
* a token whose request, position or page lies outside the table or the pool
  writes nothing.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0


def e4m3_encode(x) -> np.ndarray:
    """Float32 values -> OCP E4M3 ("fn") codes (uint8): round to nearest, ties
    to even, saturating at +-448; NaN stays NaN.  The rounding itself is torch's
    float8_e4m3fn cast (a library routine); the clamp first makes it saturate
    (torch alone turns values from 480 on into NaN)."""
    x = torch.as_tensor(np.asarray(x, dtype=np.float32))
    y = torch.where(torch.isnan(x), x, x.clamp(-E4M3_MAX, E4M3_MAX))
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _valid_slot(b, pos, kv_indptr, kv_page_indices, page_size, num_pages):
    if b < 0 or b + 1 >= len(kv_indptr) or pos < 0:
        return None
    beg, end = int(kv_indptr[b]), int(kv_indptr[b + 1])
    pi = pos // page_size
    if pi >= end - beg:
        return None
    page = int(kv_page_indices[beg + pi])
    if page < 0 or page >= num_pages:
        return None
    return page, pos % page_size


def append_kv(k_cache, v_cache, k_new, v_new, batch_indices, positions, kv_indptr, kv_page_indices,
              page_size: int, k_scale=None, v_scale=None):
    """Return (k_cache', v_cache', n_skipped): copies of the pools (torch tensors
    [num_pages, page_size, Hk, D] in the pool dtype, moved to the CPU) with the
    new rows written, one token at a time in index order."""
    k = k_cache.detach().cpu().clone()
    v = v_cache.detach().cpu().clone()
    kn = k_new.detach().cpu().float().numpy()
    vn = v_new.detach().cpu().float().numpy()
    bi = np.asarray(batch_indices.cpu() if torch.is_tensor(batch_indices) else batch_indices, dtype=np.int64)
    ps = np.asarray(positions.cpu() if torch.is_tensor(positions) else positions, dtype=np.int64)
    indptr = np.asarray(kv_indptr.cpu() if torch.is_tensor(kv_indptr) else kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_page_indices.cpu() if torch.is_tensor(kv_page_indices) else kv_page_indices,
                     dtype=np.int64)
    fp8 = k.dtype == torch.float8_e4m3fn
    if fp8:
        ks = np.asarray(k_scale.detach().cpu(), dtype=np.float32)
        vs = np.asarray(v_scale.detach().cpu(), dtype=np.float32)
        k8, v8 = k.view(torch.uint8).numpy(), v.view(torch.uint8).numpy()
    skipped = 0
    for i in range(len(bi)):
        where = _valid_slot(int(bi[i]), int(ps[i]), indptr, idx, page_size, k.shape[0])
        if where is None:
            skipped += 1
            continue
        page, slot = where
        if fp8:
            for h in range(k.shape[2]):
                k8[page, slot, h] = e4m3_encode(kn[i, h].astype(np.float32) / ks[h])
                v8[page, slot, h] = e4m3_encode(vn[i, h].astype(np.float32) / vs[h])
        else:
            k[page, slot] = k_new[i].detach().cpu().to(k.dtype)
            v[page, slot] = v_new[i].detach().cpu().to(v.dtype)
    return k, v, skipped
