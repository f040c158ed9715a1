"""Seeded synthetic inputs for batched paged-KV decode attention.

This module builds inputs only: page tables (CSR ``kv_indptr`` /
``kv_page_indices`` / ``kv_last_page_len``), a paged K/V pool in the NHD
layout ``[num_pages, page_size, num_kv_heads, head_dim]``, queries, and, for an
fp8 pool, the per-kv-head fp32 scales.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle may consume what it
produces.

The shapes follow the workloads named on the FlashInfer pages: the quickstart
``single_decode_with_kv_cache`` shapes (q ``[32, 128]``, K/V ``[2048, 32, 128]``
fp16, page 1 "Getting started", step 4), the paged pool of the deep-dive page
("The Code, Annotated", snippet one: page_size 16, pages drawn from a pool much
larger than one batch), GQA decode at batch 64 (page 2, "What the project
publishes about performance"), and cascade decode of a batch sharing one long
prompt (page 2, "Cascade attention for shared prefixes").  The serving
benchmarks those pages measure on are not available; these seeded inputs of the
same shapes stand in for them.

Random choices: lengths and page placement come from
``numpy.random.default_rng(seed)``; tensor values come from a
``torch.Generator`` seeded with the same seed on the target device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

__all__ = [
    "PagedBatch",
    "make_paged",
    "make_config",
    "CONFIG_NAMES",
    "lengths_to_page_table",
]

_TORCH_DTYPES = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "e4m3": torch.float8_e4m3fn,
}

# E4M3 (OCP FP8, "fn" variant) largest finite magnitude.
_E4M3_MAX = 448.0

CONFIG_NAMES = {
    1: "single_request_f16_h32_l2048_p16",
    2: "batch64_gqa4_bf16_l512to4096_p16",
    3: "batch128_gqa8_bf16_skewed_p16",
    4: "cascade256_gqa4_bf16_prefix8192_suffix128to512_p16",
    5: "batch16_gqa8_e4m3kv_l131072_p64",
}


@dataclass
class PagedBatch:
    """One decode batch over a paged KV pool.

    Attributes mirror the plan/run arguments: ``kv_indptr[b]..kv_indptr[b+1]``
    indexes request b's physical pages in ``kv_page_indices``; the last page of
    request b holds ``kv_last_page_len[b]`` valid tokens (1..page_size).
    """

    name: str
    q: torch.Tensor  # [B, Hq, D]
    k_cache: torch.Tensor  # [num_pages, P, Hk, D]
    v_cache: torch.Tensor  # [num_pages, P, Hk, D]
    kv_indptr: np.ndarray  # int32 [B+1]
    kv_page_indices: np.ndarray  # int32 [nnz]
    kv_last_page_len: np.ndarray  # int32 [B]
    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    sm_scale: float
    k_scale: Optional[torch.Tensor] = None  # fp32 [Hk] for an e4m3 pool
    v_scale: Optional[torch.Tensor] = None
    kv_lens: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    # cascade: one shared prefix page list, attended by every request
    prefix_page_indices: Optional[np.ndarray] = None
    prefix_last_page_len: int = 0
    # prefix tree: shared levels, outermost first, each
    # (req_indptr, kv_indptr, kv_page_indices, kv_last_page_len) over its nodes
    levels: Optional[list] = None
    # prefill: request r's query tokens are q[qo_indptr[r] .. qo_indptr[r+1]-1]
    qo_indptr: Optional[np.ndarray] = None

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.shape[0] - 1)

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def prefix_len(self) -> int:
        if self.prefix_page_indices is None or len(self.prefix_page_indices) == 0:
            return 0
        return (len(self.prefix_page_indices) - 1) * self.page_size + self.prefix_last_page_len

    def to(self, device) -> "PagedBatch":
        out = PagedBatch(**{k: getattr(self, k) for k in self.__dataclass_fields__})
        out.q = self.q.to(device)
        out.k_cache = self.k_cache.to(device)
        out.v_cache = self.v_cache.to(device)
        if self.k_scale is not None:
            out.k_scale = self.k_scale.to(device)
            out.v_scale = self.v_scale.to(device)
        return out


def lengths_to_page_table(lengths: Sequence[int], page_size: int, page_order: np.ndarray):
    """CSR page table for requests of the given token counts.

    Request b gets ``ceil(L_b / page_size)`` consecutive entries of
    ``page_order``; its last page holds ``L_b - (n_b - 1) * page_size`` tokens
    (``L_b mod page_size``, or ``page_size`` when that is 0).  A request of
    length 0 gets no page and a last_page_len of 0.
    """
    lengths = np.asarray(lengths, dtype=np.int64)
    n_pages = (lengths + page_size - 1) // page_size
    indptr = np.zeros(len(lengths) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(n_pages)
    nnz = int(indptr[-1])
    if nnz > len(page_order):
        raise ValueError(f"pool too small: need {nnz} pages, have {len(page_order)}")
    indices = np.asarray(page_order[:nnz], dtype=np.int32)
    last = np.where(n_pages > 0, lengths - (n_pages - 1) * page_size, 0)
    return indptr.astype(np.int32), indices, last.astype(np.int32)


def _randn(shape, gen: torch.Generator, device, dtype) -> torch.Tensor:
    """N(0,1) values rounded (RNE) to ``dtype``; generated in fp32 by slabs."""
    out = torch.empty(shape, dtype=dtype, device=device)
    rows = shape[0]
    per_row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    slab = max(1, (1 << 26) // max(per_row, 1))
    for r0 in range(0, rows, slab):
        r1 = min(rows, r0 + slab)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen,
                                 device=device, dtype=torch.float32).to(dtype)
    return out


def _quantize_e4m3_per_head(x32: torch.Tensor):
    """Per-kv-head symmetric e4m3 quantisation of a ``[N, P, Hk, D]`` fp32 pool.

    scale[h] = amax(|x[:, :, h, :]|) / 448; stored value = e4m3(x / scale[h])
    (round to nearest even, clamped to the finite range).  Returns
    ``(codes as torch.float8_e4m3fn, scale fp32 [Hk])``.
    """
    amax = x32.abs().amax(dim=(0, 1, 3)).to(torch.float32)
    scale = torch.where(amax > 0, amax / _E4M3_MAX, torch.ones_like(amax))
    codes = torch.empty(x32.shape, dtype=torch.float8_e4m3fn, device=x32.device)
    n = x32.shape[0]
    slab = max(1, (1 << 26) // max(int(np.prod(x32.shape[1:])), 1))
    for r0 in range(0, n, slab):
        r1 = min(n, r0 + slab)
        y = (x32[r0:r1] / scale.view(1, 1, -1, 1)).clamp_(-_E4M3_MAX, _E4M3_MAX)
        codes[r0:r1] = y.to(torch.float8_e4m3fn)
    return codes, scale


def make_paged(
    *,
    seed: int,
    lengths: Sequence[int],
    num_qo_heads: int,
    num_kv_heads: int,
    head_dim: int = 128,
    page_size: int = 16,
    q_dtype: str = "bf16",
    kv_dtype: str = "bf16",
    pool_pages: Optional[int] = None,
    identity_pages: bool = False,
    device="cpu",
    name: str = "custom",
    prefix_len: int = 0,
    sm_scale: Optional[float] = None,
    pool_layout: str = "split",
) -> PagedBatch:
    """Build a seeded paged decode batch.

    ``lengths`` are per-request token counts (of the private part when
    ``prefix_len`` > 0).  Pages are placed by a seeded random permutation of the
    pool unless ``identity_pages``.  With ``prefix_len`` > 0 the first
    ``ceil(prefix_len / page_size)`` pages of the permutation form one shared
    prefix list.  ``pool_layout="interleaved"`` stores the pool as
    ``[num_pages, 2, P, Hk, D]`` (K at index 0, V at 1) and returns K and V as
    strided views of it, like the combined pool of the deep-dive page.
    """
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    P = page_size
    prefix_pages = (prefix_len + P - 1) // P
    need = int(((lengths + P - 1) // P).sum()) + prefix_pages
    if pool_pages is None:
        pool_pages = max(need, 1)
    if need > pool_pages:
        raise ValueError(f"pool of {pool_pages} pages cannot hold {need}")
    order = np.arange(pool_pages, dtype=np.int64) if identity_pages else rng.permutation(pool_pages)
    prefix_idx = None
    prefix_last = 0
    if prefix_pages:
        prefix_idx = np.asarray(order[:prefix_pages], dtype=np.int32)
        prefix_last = prefix_len - (prefix_pages - 1) * P
        order = order[prefix_pages:]
    indptr, indices, last = lengths_to_page_table(lengths, P, order)

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B = len(lengths)
    q = _randn((B, num_qo_heads, head_dim), gen, device, _TORCH_DTYPES[q_dtype])
    shape = (pool_pages, P, num_kv_heads, head_dim)
    k_scale = v_scale = None
    if kv_dtype == "e4m3":
        k32 = _randn(shape, gen, device, torch.float32)
        k_cache, k_scale = _quantize_e4m3_per_head(k32)
        del k32
        v32 = _randn(shape, gen, device, torch.float32)
        v_cache, v_scale = _quantize_e4m3_per_head(v32)
        del v32
    else:
        dt = _TORCH_DTYPES[kv_dtype]
        if pool_layout == "interleaved":
            pool = torch.empty((pool_pages, 2) + shape[1:], dtype=dt, device=device)
            pool[:, 0] = _randn(shape, gen, device, dt)
            pool[:, 1] = _randn(shape, gen, device, dt)
            k_cache, v_cache = pool[:, 0], pool[:, 1]
        else:
            k_cache = _randn(shape, gen, device, dt)
            v_cache = _randn(shape, gen, device, dt)
    return PagedBatch(
        name=name,
        q=q,
        k_cache=k_cache,
        v_cache=v_cache,
        kv_indptr=indptr,
        kv_page_indices=indices,
        kv_last_page_len=last,
        page_size=P,
        num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else float(sm_scale),
        k_scale=k_scale,
        v_scale=v_scale,
        kv_lens=lengths.astype(np.int32),
        prefix_page_indices=prefix_idx,
        prefix_last_page_len=int(prefix_last),
    )


def make_tree(*, seed: int, levels: Sequence[Tuple[Sequence[int], Sequence[int]]], lengths: Sequence[int],
              num_qo_heads: int, num_kv_heads: int, head_dim: int = 128, page_size: int = 16,
              q_dtype: str = "bf16", kv_dtype: str = "bf16", device="cpu", name: str = "tree") -> PagedBatch:
    """A decode batch over a prefix tree: ``levels`` lists the shared levels,
    outermost first, as (requests per node, tokens per node); each level's
    request counts sum to the batch (``len(lengths)``), node n serving the
    next ``count[n]`` requests in order.  ``lengths`` are the requests' own
    (suffix) token counts.  All pages of all levels and of the suffixes are
    placed by one seeded permutation of the pool."""
    B = len(lengths)
    P = page_size
    need = sum(int(((np.asarray(toks, np.int64) + P - 1) // P).sum()) for _, toks in levels)
    base = make_paged(seed=seed, lengths=lengths, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                      head_dim=head_dim, page_size=P, q_dtype=q_dtype, kv_dtype=kv_dtype, device=device,
                      name=name, pool_pages=int(((np.asarray(lengths, np.int64) + P - 1) // P).sum()) + need)
    # the suffix tables use the first pages of make_paged's permutation; the
    # levels take the pages it left over, in a second seeded order
    used = set(np.asarray(base.kv_page_indices, np.int64).tolist())
    free = np.asarray([p for p in range(base.num_pages) if p not in used], np.int64)
    free = np.random.default_rng(seed + 1).permutation(free)
    out_levels = []
    off = 0
    for counts, toks in levels:
        counts = np.asarray(counts, np.int64)
        if counts.sum() != B or np.any(counts < 0):
            raise ValueError("each level's request counts must sum to the batch")
        req_indptr = np.zeros(len(counts) + 1, np.int32)
        req_indptr[1:] = np.cumsum(counts)
        ip, idx, last = lengths_to_page_table(toks, P, free[off:])
        off += int(ip[-1])
        out_levels.append((req_indptr, ip, idx, last))
    base.levels = out_levels
    return base


def make_prefill(*, seed: int, q_lens: Sequence[int], kv_lens: Sequence[int], num_qo_heads: int,
                 num_kv_heads: int, head_dim: int = 128, page_size: int = 16, q_dtype: str = "bf16",
                 kv_dtype: str = "bf16", device="cpu", name: str = "prefill") -> PagedBatch:
    """A prefill / append batch: request r has ``kv_lens[r]`` keys in its pages
    (its new tokens' keys included) and ``q_lens[r] <= kv_lens[r]`` query
    tokens, stacked into q ``[sum(q_lens), Hq, D]``."""
    q_lens = np.asarray(q_lens, np.int64)
    kv_lens = np.asarray(kv_lens, np.int64)
    if np.any(q_lens > kv_lens) or np.any(q_lens < 0):
        raise ValueError("0 <= q_len <= kv_len per request")
    b = make_paged(seed=seed, lengths=kv_lens, num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads,
                   head_dim=head_dim, page_size=page_size, q_dtype=q_dtype, kv_dtype=kv_dtype, device=device,
                   name=name)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7)
    T = int(q_lens.sum())
    b.q = _randn((max(T, 0), num_qo_heads, head_dim), gen, device, _TORCH_DTYPES[q_dtype])
    qo = np.zeros(len(q_lens) + 1, np.int32)
    qo[1:] = np.cumsum(q_lens)
    b.qo_indptr = qo
    return b


TREE_WORKLOAD = "tree3_b256_root4096_16x1024_suffix64to512_gqa4_bf16_p16"
PREFILL_WORKLOAD = "prefill_b16_q512_kv1024to4096_gqa4_bf16_p16"


def make_config_tree(device="cpu", batch: Optional[int] = None) -> PagedBatch:
    """Prefix-tree decode workload: 256 requests (or ``batch``, a multiple of
    16) under one 4096-key root, 16 branches of 1024 keys (16 requests each)
    and their own 64-512 keys; GQA 32/8, bf16, page 16 (the cascade
    workload's shapes, with one more shared level)."""
    B = batch or 256
    rng = np.random.default_rng(2001)
    lengths = rng.integers(64, 512, size=B, endpoint=True)
    return make_tree(seed=2001, levels=[([B], [4096]), ([B // 16] * 16, [1024] * 16)], lengths=lengths,
                     num_qo_heads=32, num_kv_heads=8, page_size=16, device=device, name=TREE_WORKLOAD)


def make_config_prefill(device="cpu", batch: Optional[int] = None) -> PagedBatch:
    """Append-prefill workload: 16 requests (or ``batch``), 512 new tokens
    each on top of 512-3584 cached ones (1024-4096 keys in all, the new
    tokens' included); GQA 32/8, bf16, page 16."""
    B = batch or 16
    rng = np.random.default_rng(2002)
    kv = rng.integers(1024, 4096, size=B, endpoint=True)
    return make_prefill(seed=2002, q_lens=[512] * B, kv_lens=kv, num_qo_heads=32, num_kv_heads=8, page_size=16,
                        device=device, name=PREFILL_WORKLOAD)


@dataclass
class MlaBatch:
    """One MLA decode batch: latent cache ckv ``[N, P, 512]`` and rotary key
    cache kpe ``[N, P, 64]`` (one latent "kv head" shared by all query heads),
    queries q_nope ``[B, H, 512]`` (already in the latent space) and q_pe
    ``[B, H, 64]``, and a CSR page table as for ``PagedBatch``."""

    name: str
    q_nope: torch.Tensor
    q_pe: torch.Tensor
    ckv_cache: torch.Tensor
    kpe_cache: torch.Tensor
    kv_indptr: np.ndarray
    kv_page_indices: np.ndarray
    kv_last_page_len: np.ndarray
    page_size: int
    num_heads: int
    sm_scale: float
    kv_lens: np.ndarray

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.shape[0] - 1)


MLA_WORKLOAD = "mla_b64_h128_l3072to8192_latent512_rope64_bf16_p16"


def make_mla(*, seed: int, lengths: Sequence[int], num_heads: int = 128, page_size: int = 16,
             pool_pages: Optional[int] = None, device="cpu", name: str = "mla",
             sm_scale: Optional[float] = None) -> MlaBatch:
    """Seeded MLA decode batch (bf16, N(0,1) values).  ``sm_scale`` defaults to
    1/sqrt(128 + 64), the query-key width of the decompressed heads (128
    no-RoPE + 64 RoPE dimensions)."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    P = page_size
    need = int(((lengths + P - 1) // P).sum())
    pool_pages = max(need, 1) if pool_pages is None else pool_pages
    order = rng.permutation(pool_pages)
    indptr, indices, last = lengths_to_page_table(lengths, P, order)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    B = len(lengths)
    bf = torch.bfloat16
    return MlaBatch(
        name=name,
        q_nope=_randn((B, num_heads, 512), gen, device, bf),
        q_pe=_randn((B, num_heads, 64), gen, device, bf),
        ckv_cache=_randn((pool_pages, P, 512), gen, device, bf),
        kpe_cache=_randn((pool_pages, P, 64), gen, device, bf),
        kv_indptr=indptr, kv_page_indices=indices, kv_last_page_len=last, page_size=P, num_heads=num_heads,
        sm_scale=(1.0 / math.sqrt(192.0)) if sm_scale is None else float(sm_scale),
        kv_lens=lengths.astype(np.int32))


def make_config_mla(device="cpu", batch: Optional[int] = None) -> MlaBatch:
    """The deep dive's DeepSeek-V3 serving step: 64 concurrent decode requests
    (or ``batch``) of 3072-8192 cached tokens, 128 query heads, latent 512 +
    RoPE 64, bf16, page 16."""
    B = batch or 64
    rng = np.random.default_rng(3003)
    lengths = rng.integers(3072, 8192, size=B, endpoint=True)
    return make_mla(seed=3003, lengths=lengths, num_heads=128, page_size=16, device=device, name=MLA_WORKLOAD)


def config_lengths(idx: int, batch: Optional[int] = None) -> np.ndarray:
    """Per-request token counts of the five standard workloads (seeded)."""
    rng = np.random.default_rng(1000 + idx)
    if idx == 1:
        return np.array([2048], dtype=np.int64)
    if idx == 2:
        return rng.integers(512, 4096, size=batch or 64, endpoint=True)
    if idx == 3:
        n = batch or 128
        rest = np.clip(np.rint(rng.lognormal(math.log(600.0), 0.8, size=max(n - 8, 0))), 16, 4096)
        lens = np.concatenate([[32768], [8192] * 7, rest]).astype(np.int64)[:n]
        return lens[rng.permutation(len(lens))]
    if idx == 4:
        return rng.integers(128, 512, size=batch or 256, endpoint=True)
    if idx == 5:
        return np.full(batch or 16, 131072, dtype=np.int64)
    raise ValueError(idx)


def config_geometry(idx: int):
    """(page_size, num_qo_heads, num_kv_heads, q dtype, kv dtype) of a standard workload."""
    return {1: (16, 32, 32, "f16", "f16"), 2: (16, 32, 8, "bf16", "bf16"), 3: (16, 64, 8, "bf16", "bf16"),
            4: (16, 32, 8, "bf16", "bf16"), 5: (64, 64, 8, "bf16", "e4m3")}[idx]


def make_config(idx: int, device="cpu", batch: Optional[int] = None) -> PagedBatch:
    """The five standard workloads.  ``batch`` shrinks the request count (for
    tests that keep a config's structure at a size the oracle finishes fast)."""
    lens = config_lengths(idx, batch)
    name = CONFIG_NAMES[idx] + ("" if batch is None else f"_b{batch}")
    if idx == 1:
        return make_paged(seed=1, lengths=lens, num_qo_heads=32, num_kv_heads=32, page_size=16,
                          q_dtype="f16", kv_dtype="f16", identity_pages=True, device=device,
                          name=name)
    if idx == 2:
        return make_paged(seed=2, lengths=lens, num_qo_heads=32, num_kv_heads=8, page_size=16,
                          pool_pages=20000 if batch is None else None, device=device, name=name)
    if idx == 3:
        need = int(((lens + 15) // 16).sum())
        return make_paged(seed=3, lengths=lens, num_qo_heads=64, num_kv_heads=8, page_size=16,
                          pool_pages=40000 if batch is None else max(need, 1), device=device,
                          name=name)
    if idx == 4:
        need = 512 + int(((lens + 15) // 16).sum())
        return make_paged(seed=4, lengths=lens, num_qo_heads=32, num_kv_heads=8, page_size=16,
                          pool_pages=need + need // 4, prefix_len=8192, device=device, name=name)
    if idx == 5:
        need = int(((lens + 63) // 64).sum())
        return make_paged(seed=5, lengths=lens, num_qo_heads=64, num_kv_heads=8, page_size=64,
                          q_dtype="bf16", kv_dtype="e4m3",
                          pool_pages=32768 if batch is None else need, device=device, name=name)
    raise ValueError(idx)


def cascade_as_plain(batch: PagedBatch) -> PagedBatch:
    """The same cascade batch expressed as one page list per request
    (shared prefix pages followed by the request's own pages).  Valid only when
    the prefix's last page is full, which the standard cascade workload has."""
    assert batch.prefix_page_indices is not None
    assert batch.prefix_last_page_len == batch.page_size
    pre = batch.prefix_page_indices
    B = batch.batch
    lists = []
    for b in range(B):
        own = batch.kv_page_indices[batch.kv_indptr[b]:batch.kv_indptr[b + 1]]
        lists.append(np.concatenate([pre, own]))
    indptr = np.zeros(B + 1, dtype=np.int32)
    indptr[1:] = np.cumsum([len(x) for x in lists])
    out = PagedBatch(**{k: getattr(batch, k) for k in batch.__dataclass_fields__})
    out.kv_indptr = indptr
    out.kv_page_indices = np.concatenate(lists).astype(np.int32)
    out.kv_last_page_len = batch.kv_last_page_len.copy()
    out.kv_lens = batch.kv_lens + batch.prefix_len
    out.prefix_page_indices = None
    out.prefix_last_page_len = 0
    return out
