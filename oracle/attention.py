"""fp64 CPU oracle for batched paged-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA path.

What it computes is the plain definition of decode attention over a paged
(CSR page-table) KV cache, written out in float64:

* Page table walk (FlashInfer deep dive, snackonai.com, "The Code, Annotated",
  snippet one: ``indptr`` / ``indices`` / ``last_page_len`` and the pool
  ``[num_pages, (K,V), page_size, heads, head_dim]`` in the NHD layout): request
  b owns pages ``indices[indptr[b]:indptr[b+1]]`` in that order; every page is
  full except the last, which holds ``last_page_len[b]`` tokens.
* Decode attention for one query token (ai-tldr.dev tool card, "Getting
  started", step 4, ``single_decode_with_kv_cache``: q ``[num_qo_heads,
  head_dim]``, K/V ``[kv_len, num_kv_heads, head_dim]``):
  ``s_j = sm_scale * <q_h, k_j>``, ``lse = log sum_j exp(s_j)`` (natural log),
  ``o_h = sum_j exp(s_j - lse) v_j``.  Grouped-query heads map contiguously:
  qo head h reads kv head ``h // (Hq / Hk)``.
* Attention states and their merge (aquanode.io 2026 guide, "Cascade attention
  for shared prefixes": merge_state / merge_states in flashinfer.cascade): a
  state is ``(o, lse)``; the merge of two states over disjoint key sets is the
  state over their union.
* Cascade decode (same section; deep dive, "Why This Design Works": the shared
  prefix is read once but counted as if each request owns it): the prefix state
  merged with each request's own state; over a prefix tree, one state per
  level merged with the request's own.
* Prefill / append attention (README mirror, "Core Features"): several query
  tokens per request, each at the end of its sequence, attending the keys up to
  its own position (causal) or all keys.

Readings where the pages are silent (each is also listed in the design notes):
natural-log LSE; ``sm_scale`` defaults to ``1/sqrt(head_dim)``; an empty key
set has ``o = 0`` and ``lse = -inf``; fp8 pool values are multiplied by their
per-kv-head fp32 scale in float64.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

try:  # torch is only used to turn bf16 / fp8 tensors into float64 exactly
    import torch
except Exception:  # pragma: no cover
    torch = None

__all__ = [
    "to_f64",
    "request_tokens",
    "gather_kv",
    "attend",
    "paged_decode",
    "single_decode",
    "merge_state",
    "merge_states",
    "cascade_decode",
    "multilevel_cascade_decode",
    "paged_prefill",
]


def to_f64(x) -> np.ndarray:
    """Exact float64 copy of a numpy array or a CPU torch tensor of any float type."""
    if torch is not None and isinstance(x, torch.Tensor):
        return x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def request_tokens(kv_indptr, kv_page_indices, kv_last_page_len, page_size: int, b: int):
    """The (physical page, slot) of every key of request b, in sequence order.

    Deep dive, "The Code, Annotated", snippet one: request b's pages are
    ``indices[indptr[b] .. indptr[b+1]-1]``; all are full but the last, which
    holds ``last_page_len[b]`` tokens.
    """
    start, end = int(kv_indptr[b]), int(kv_indptr[b + 1])
    out = []
    for i in range(start, end):
        page = int(kv_page_indices[i])
        n = int(kv_last_page_len[b]) if i == end - 1 else page_size
        for t in range(n):
            out.append((page, t))
    return out


def _take_pages(cache, pages):
    """``cache[pages]`` for a numpy array or a CPU torch tensor (no dtype change)."""
    if torch is not None and isinstance(cache, torch.Tensor):
        return cache[torch.as_tensor(pages, dtype=torch.long)]
    return np.asarray(cache)[pages]


def gather_kv(cache: np.ndarray, tokens: Sequence[Tuple[int, int]]) -> np.ndarray:
    """Stack ``cache[page, slot]`` (shape ``[Hk, D]``) for the given tokens -> ``[L, Hk, D]``."""
    if len(tokens) == 0:
        return np.zeros((0,) + cache.shape[2:], dtype=np.float64)
    pages = np.fromiter((p for p, _ in tokens), dtype=np.int64, count=len(tokens))
    slots = np.fromiter((t for _, t in tokens), dtype=np.int64, count=len(tokens))
    return cache[pages, slots]


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float):
    """Attention of one query vector over ``k, v`` of shape ``[L, D]``.

    Returns ``(o [D], lse)`` with ``s_j = sm_scale * <q, k_j>``,
    ``lse = m + ln sum_j exp(s_j - m)`` for ``m = max_j s_j`` and
    ``o = sum_j exp(s_j - lse) v_j``.  An empty key set gives ``(0, -inf)``.
    """
    if k.shape[0] == 0:
        return np.zeros(v.shape[1], dtype=np.float64), -math.inf
    s = sm_scale * (k @ q)
    m = float(np.max(s))
    lse = m + math.log(float(np.sum(np.exp(s - m))))
    w = np.exp(s - lse)
    return w @ v, lse


def paged_decode(
    q,
    k_cache,
    v_cache,
    kv_indptr,
    kv_page_indices,
    kv_last_page_len,
    *,
    sm_scale: Optional[float] = None,
    k_scale=None,
    v_scale=None,
    rows: Optional[Iterable[Tuple[int, int]]] = None,
):
    """Batched decode attention over a paged KV cache.

    q ``[B, Hq, D]``; caches ``[num_pages, P, Hk, D]`` (any float dtype, or fp8
    with ``k_scale`` / ``v_scale`` of shape ``[Hk]``).  Returns
    ``(o [B, Hq, D], lse [B, Hq])`` in float64.  With ``rows`` (pairs
    ``(b, h)``) only those outputs are computed; the others are NaN.
    """
    qf = to_f64(q)
    B, Hq, D = qf.shape
    P, Hk = int(k_cache.shape[1]), int(k_cache.shape[2])
    if Hq % Hk != 0:
        raise ValueError("num_qo_heads must be a multiple of num_kv_heads")
    g = Hq // Hk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    ks = None if k_scale is None else to_f64(k_scale)
    vs = None if v_scale is None else to_f64(v_scale)
    want = None
    if rows is not None:
        want = {}
        for b, h in rows:
            want.setdefault(int(b), set()).add(int(h))
    o = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    for b in range(B):
        if want is not None and b not in want:
            continue
        toks = request_tokens(kv_indptr, kv_page_indices, kv_last_page_len, P, b)
        if toks:
            pages = sorted({p for p, _ in toks})
            # convert only the pages this request touches
            remap = {p: i for i, p in enumerate(pages)}
            kp = to_f64(_take_pages(k_cache, pages))
            vp = to_f64(_take_pages(v_cache, pages))
            local = [(remap[p], t) for p, t in toks]
            kb = gather_kv(kp, local)
            vb = gather_kv(vp, local)
        else:
            kb = np.zeros((0, Hk, D))
            vb = np.zeros((0, Hk, D))
        if ks is not None:
            kb = kb * ks[None, :, None]
        if vs is not None:
            vb = vb * vs[None, :, None]
        heads = range(Hq) if want is None else sorted(want[b])
        for h in heads:
            kvh = h // g
            o[b, h], lse[b, h] = attend(qf[b, h], kb[:, kvh, :], vb[:, kvh, :], sm_scale)
    return o, lse


def single_decode(q, k, v, *, sm_scale: Optional[float] = None, k_scale=None, v_scale=None):
    """Quickstart shapes: q ``[Hq, D]``, contiguous K/V ``[L, Hk, D]`` -> ``(o [Hq, D], lse [Hq])``."""
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    Hq, D = qf.shape
    Hk = kf.shape[1]
    g = Hq // Hk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    if k_scale is not None:
        kf = kf * to_f64(k_scale)[None, :, None]
    if v_scale is not None:
        vf = vf * to_f64(v_scale)[None, :, None]
    o = np.zeros((Hq, D))
    lse = np.zeros(Hq)
    for h in range(Hq):
        o[h], lse[h] = attend(qf[h], kf[:, h // g, :], vf[:, h // g, :], sm_scale)
    return o, lse


def merge_state(v_a, s_a, v_b, s_b):
    """Merge two attention states over disjoint key sets (flashinfer.cascade merge_state).

    ``s = max(s_a, s_b) + ln(exp(s_a - max) + exp(s_b - max))`` and
    ``v = v_a exp(s_a - s) + v_b exp(s_b - s)``, elementwise over the leading
    dimensions of ``s``; ``v`` has one more trailing dimension (head_dim).  A
    state with ``s = -inf`` is empty: merging with it is the identity, and two
    empty states merge to ``(0, -inf)``.
    """
    va, vb = to_f64(v_a), to_f64(v_b)
    sa, sb = to_f64(s_a), to_f64(s_b)
    m = np.maximum(sa, sb)
    both_empty = np.isneginf(m)
    m_safe = np.where(both_empty, 0.0, m)
    ea = np.where(np.isneginf(sa), 0.0, np.exp(sa - m_safe))
    eb = np.where(np.isneginf(sb), 0.0, np.exp(sb - m_safe))
    tot = ea + eb
    s = np.where(both_empty, -np.inf, m_safe + np.log(np.where(both_empty, 1.0, tot)))
    wa = np.where(both_empty, 0.0, ea / np.where(both_empty, 1.0, tot))
    wb = np.where(both_empty, 0.0, eb / np.where(both_empty, 1.0, tot))
    v = va * wa[..., None] + vb * wb[..., None]
    return v, s


def merge_states(v, s):
    """Merge k states: v ``[n, k, H, D]``, s ``[n, k, H]`` -> ``([n, H, D], [n, H])``, left fold."""
    vf, sf = to_f64(v), to_f64(s)
    n, k = sf.shape[0], sf.shape[1]
    acc_v = np.zeros((n,) + vf.shape[2:])
    acc_s = np.full((n,) + sf.shape[2:], -np.inf)
    for i in range(k):
        acc_v, acc_s = merge_state(acc_v, acc_s, vf[:, i], sf[:, i])
    return acc_v, acc_s


def cascade_decode(
    q,
    k_cache,
    v_cache,
    prefix_page_indices,
    prefix_last_page_len: int,
    kv_indptr,
    kv_page_indices,
    kv_last_page_len,
    *,
    sm_scale: Optional[float] = None,
    k_scale=None,
    v_scale=None,
    rows=None,
):
    """Shared-prefix decode: every request attends the one prefix page list and
    its own page list; the two states are merged per (request, qo head)."""
    B = to_f64(q).shape[0]
    pre = np.asarray(prefix_page_indices, dtype=np.int64)
    n_pre = len(pre)
    pre_indptr = np.arange(B + 1, dtype=np.int64) * n_pre
    pre_idx = np.tile(pre, B)
    pre_last = np.full(B, prefix_last_page_len if n_pre else 0, dtype=np.int64)
    o_p, s_p = paged_decode(q, k_cache, v_cache, pre_indptr, pre_idx, pre_last,
                            sm_scale=sm_scale, k_scale=k_scale, v_scale=v_scale, rows=rows)
    o_s, s_s = paged_decode(q, k_cache, v_cache, kv_indptr, kv_page_indices, kv_last_page_len,
                            sm_scale=sm_scale, k_scale=k_scale, v_scale=v_scale, rows=rows)
    return merge_state(o_p, s_p, o_s, s_s)


def _expand_level(req_indptr, kv_indptr, kv_page_indices, kv_last_page_len, batch: int):
    """Per-request page table of one shared level: request b in node n (the
    nodes' request ranges ``req_indptr[n] .. req_indptr[n+1]-1`` partition the
    batch) owns node n's pages."""
    req_indptr = np.asarray(req_indptr, dtype=np.int64)
    kv_indptr = np.asarray(kv_indptr, dtype=np.int64)
    idx = np.asarray(kv_page_indices, dtype=np.int64)
    last = np.asarray(kv_last_page_len, dtype=np.int64)
    if req_indptr[0] != 0 or req_indptr[-1] != batch or np.any(np.diff(req_indptr) < 0):
        raise ValueError("the nodes' request ranges must partition the batch")
    out_indptr = [0]
    out_idx = []
    out_last = np.zeros(batch, dtype=np.int64)
    for n in range(len(req_indptr) - 1):
        pages = idx[kv_indptr[n]:kv_indptr[n + 1]]
        for b in range(req_indptr[n], req_indptr[n + 1]):
            out_idx.extend(pages.tolist())
            out_indptr.append(out_indptr[-1] + len(pages))
            out_last[b] = last[n] if len(pages) else 0
    return np.asarray(out_indptr, np.int64), np.asarray(out_idx, np.int64), out_last


def multilevel_cascade_decode(q, k_cache, v_cache, levels, kv_indptr, kv_page_indices, kv_last_page_len, *,
                              sm_scale: Optional[float] = None, k_scale=None, v_scale=None, rows=None):
    """Cascade decode over a prefix tree (2026 guide, "Cascade attention for
    shared prefixes"; README mirror, "Core Features": cascade attention as a
    hierarchical KV cache for shared prefixes).

    ``levels`` lists the shared levels, outermost first, each as
    ``(req_indptr, kv_indptr, kv_page_indices, kv_last_page_len)``: node n of
    the level serves requests ``req_indptr[n] .. req_indptr[n+1]-1`` (the
    nodes partition the batch) and owns pages ``kv_page_indices[kv_indptr[n]
    .. kv_indptr[n+1]-1`` (all full but the last).  The last three arguments
    are each request's own pages, as for ``paged_decode``.  Each request's
    state over every level's keys and its own is the merge of the per-level
    states (merge_state over disjoint key sets)."""
    B = to_f64(q).shape[0]
    acc_o = acc_s = None
    for req_indptr, ip, idx, last in levels:
        e_ip, e_idx, e_last = _expand_level(req_indptr, ip, idx, last, B)
        o_l, s_l = paged_decode(q, k_cache, v_cache, e_ip, e_idx, e_last, sm_scale=sm_scale, k_scale=k_scale,
                                v_scale=v_scale, rows=rows)
        acc_o, acc_s = (o_l, s_l) if acc_o is None else merge_state(acc_o, acc_s, o_l, s_l)
    o_s, s_s = paged_decode(q, k_cache, v_cache, kv_indptr, kv_page_indices, kv_last_page_len,
                            sm_scale=sm_scale, k_scale=k_scale, v_scale=v_scale, rows=rows)
    if acc_o is None:
        return o_s, s_s
    return merge_state(acc_o, acc_s, o_s, s_s)


def paged_prefill(q, qo_indptr, k_cache, v_cache, kv_indptr, kv_page_indices, kv_last_page_len, *,
                  causal: bool = True, sm_scale: Optional[float] = None, k_scale=None, v_scale=None,
                  rows: Optional[Iterable[Tuple[int, int]]] = None):
    """Prefill / append attention over a paged KV cache (README mirror, "Core
    Features": decode, prefill and append kernels over a paged KV cache).

    q ``[T, Hq, D]``: request r's query tokens are ``q[qo_indptr[r] ..
    qo_indptr[r+1]-1]``; its keys are all of its pages (``kv_len_r`` keys),
    the query tokens' own keys included, so token i of the request sits at
    sequence position ``kv_len_r - q_len_r + i`` and, when ``causal``, attends
    keys ``0 .. kv_len_r - q_len_r + i``; otherwise all ``kv_len_r`` keys.
    Returns ``(o [T, Hq, D], lse [T, Hq])`` in float64; with ``rows`` (pairs
    ``(token, qo head)``) only those, the rest NaN."""
    qf = to_f64(q)
    T, Hq, D = qf.shape
    P, Hk = int(k_cache.shape[1]), int(k_cache.shape[2])
    g = Hq // Hk
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    ks = None if k_scale is None else to_f64(k_scale)
    vs = None if v_scale is None else to_f64(v_scale)
    qo = np.asarray(qo_indptr, dtype=np.int64)
    want = None
    if rows is not None:
        want = {}
        for t, h in rows:
            want.setdefault(int(t), set()).add(int(h))
    o = np.full((T, Hq, D), np.nan)
    lse = np.full((T, Hq), np.nan)
    for r in range(len(qo) - 1):
        q0, q1 = int(qo[r]), int(qo[r + 1])
        if q1 == q0 or (want is not None and not any(t in want for t in range(q0, q1))):
            continue
        toks = request_tokens(kv_indptr, kv_page_indices, kv_last_page_len, P, r)
        L = len(toks)
        if L < q1 - q0:
            raise ValueError(f"request {r}: {q1 - q0} query tokens but only {L} keys")
        if toks:
            pages = sorted({p for p, _ in toks})
            remap = {p: i for i, p in enumerate(pages)}
            kp = to_f64(_take_pages(k_cache, pages))
            vp = to_f64(_take_pages(v_cache, pages))
            local = [(remap[p], t) for p, t in toks]
            kb, vb = gather_kv(kp, local), gather_kv(vp, local)
        else:
            kb = vb = np.zeros((0, Hk, D))
        if ks is not None:
            kb = kb * ks[None, :, None]
        if vs is not None:
            vb = vb * vs[None, :, None]
        for t in range(q0, q1):
            if want is not None and t not in want:
                continue
            n_keys = (L - (q1 - q0) + (t - q0) + 1) if causal else L
            heads = range(Hq) if want is None else sorted(want[t])
            for h in heads:
                kvh = h // g
                o[t, h], lse[t, h] = attend(qf[t, h], kb[:n_keys, kvh, :], vb[:n_keys, kvh, :], sm_scale)
    return o, lse
