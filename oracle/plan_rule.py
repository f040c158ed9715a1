"""Pure-Python restatement of the split-KV plan rule (integer, bit-exact).

TEST INFRASTRUCTURE ONLY: the tests compare the library's C++ planner with this
function element by element.

The pages name the goal but give no algorithm: a load-balanced, tile-based
split of requests of very different lengths over a static launch, so the plan
runs on the host before CUDA-graph capture and a replan leaves the launch shape
alone (aquanode.io 2026 guide, "What FlashInfer is", idea 3 "Load-balanced
scheduling"; deep dive, "The Architecture, Unpacked" and "It In Action", step 1).
The rule restated here is this library's reading of that goal:

1. A chunk is a run of at most 64 keys of one (request b, kv head h) row: for
   page_size P <= 64 it is ``64 // P`` whole pages, for P > 64 (a multiple of
   64) it is 64 keys inside one page.  Row (b, h) holds
   ``c_b = ceil(L_b / chunk_keys)`` chunks, ``L_b = (n_b - 1) P + last_b``.
2. Rows are ordered ``r = b * Hk + h``; their chunks, in order, form one list
   of ``W = Hk * sum_b c_b`` chunks.
3. With G CTAs, CTA c takes list positions ``[c q, (c + 1) q)`` for
   ``q = ceil(W / G)``.
4. An item is a maximal run of one row's chunks that fall to one CTA:
   ``(row, chunk_begin, chunk_end, cta)``.  Items are numbered in list order;
   an item's index is also its partial-result slot.
5. ``cta_item_begin[c]`` is the first item of CTA c (``[G]`` = item count);
   ``row_item_begin[r]`` / ``row_item_count[r]`` index each row's items.  A row
   with one item writes the final output directly; a row with two or more is
   merged by the second pass, as is a row with none (empty request).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Tuple

import numpy as np

CHUNK_KEYS = 64


def chunk_keys(page_size: int) -> int:
    if page_size <= 0:
        raise ValueError("page_size must be positive")
    if page_size <= CHUNK_KEYS:
        return (CHUNK_KEYS // page_size) * page_size
    if page_size % CHUNK_KEYS != 0:
        raise ValueError("page_size above 64 must be a multiple of 64")
    return CHUNK_KEYS


@dataclass
class Plan:
    items: np.ndarray  # int32 [n_items, 4]: row, chunk_begin, chunk_end, cta
    cta_item_begin: np.ndarray  # int32 [G + 1]
    row_item_begin: np.ndarray  # int32 [B * Hk]
    row_item_count: np.ndarray  # int32 [B * Hk]
    merge_rows: np.ndarray  # int32 [n_merge]: rows with item count != 1
    kv_len: np.ndarray  # int32 [B]
    chunk_keys: int
    quota: int


def make_plan(kv_indptr, kv_last_page_len, num_kv_heads: int, page_size: int, num_ctas: int) -> Plan:
    indptr = [int(x) for x in kv_indptr]
    last = [int(x) for x in kv_last_page_len]
    B = len(indptr) - 1
    ck = chunk_keys(page_size)
    kv_len: List[int] = []
    for b in range(B):
        n = indptr[b + 1] - indptr[b]
        kv_len.append(0 if n == 0 else (n - 1) * page_size + last[b])
    chunks = [(L + ck - 1) // ck for L in kv_len]
    W = num_kv_heads * sum(chunks)
    quota = (W + num_ctas - 1) // num_ctas if W > 0 else 0
    items: List[Tuple[int, int, int, int]] = []
    x = 0
    for b in range(B):
        for h in range(num_kv_heads):
            r = b * num_kv_heads + h
            k = 0
            while k < chunks[b]:
                cta = x // quota
                take = min(chunks[b] - k, (cta + 1) * quota - x)
                items.append((r, k, k + take, cta))
                k += take
                x += take
    n_items = len(items)
    cta_begin = []
    i = 0
    for c in range(num_ctas + 1):
        while i < n_items and items[i][3] < c:
            i += 1
        cta_begin.append(i)
    R = B * num_kv_heads
    row_begin = [0] * R
    row_count = [0] * R
    seen = [False] * R
    for idx, it in enumerate(items):
        r = it[0]
        if not seen[r]:
            row_begin[r] = idx
            seen[r] = True
        row_count[r] += 1
    for r in range(R):  # rows without items point at the next item (a valid empty range)
        if not seen[r]:
            nxt = n_items
            for idx, it in enumerate(items):
                if it[0] > r:
                    nxt = idx
                    break
            row_begin[r] = nxt
    merge_rows = [r for r in range(R) if row_count[r] != 1]
    return Plan(
        items=np.asarray(items, dtype=np.int32).reshape(-1, 4),
        cta_item_begin=np.asarray(cta_begin, dtype=np.int32),
        row_item_begin=np.asarray(row_begin, dtype=np.int32),
        row_item_count=np.asarray(row_count, dtype=np.int32),
        merge_rows=np.asarray(merge_rows, dtype=np.int32),
        kv_len=np.asarray(kv_len, dtype=np.int32),
        chunk_keys=ck,
        quota=quota,
    )
