"""CPU oracle for multi-latent attention (MLA) decode over a paged latent cache.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/`` and the measurement leg of ``bench.py`` may call it.  It shares
no code with the CUDA path.

The pages' other decode variant (deep dive, "Technical Moats": the latent KV
of DeepSeek-V2/V3 is attended without first being expanded to full K and V;
"The Code, Annotated", snippet one and "It In Action": the MLA wrapper with
``kv_lora_rank=512``, ``q_rope_dim=64``, page size 16, bf16, 128 query heads).
The pages give the shapes and the claim, not the arithmetic; the plainest
reading, used here:

* the cache holds per token a latent row ``ckv`` (512) and a rotary key part
  ``kpe`` (64), shared by every query head (one latent "kv head");
* the query of head h arrives with its no-RoPE part already multiplied into
  the latent space (``q_nope`` 512, the usual absorption of the key
  up-projection) and its rotary part ``q_pe`` (64);
* ``s_j = sm_scale * (<q_nope, ckv_j> + <q_pe, kpe_j>)``, the softmax over the
  request's keys, ``o = sum_j p_j ckv_j`` (512, still in the latent space: the
  value up-projection is applied after the kernel) and ``lse = ln sum_j
  exp(s_j)``;
* pages as in the decode oracle (CSR page table, NHD pages ``[P, 512]`` and
  ``[P, 64]``).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Tuple

import numpy as np

from oracle.attention import request_tokens, to_f64

__all__ = ["mla_decode"]


def mla_decode(q_nope, q_pe, ckv_cache, kpe_cache, kv_indptr, kv_page_indices, kv_last_page_len, *,
               sm_scale: float, rows: Optional[Iterable[Tuple[int, int]]] = None):
    """q_nope ``[B, H, 512]``, q_pe ``[B, H, 64]``; ckv_cache ``[N, P, 512]``,
    kpe_cache ``[N, P, 64]``.  Returns ``(o [B, H, 512], lse [B, H])`` in
    float64; with ``rows`` (pairs (b, h)) only those, the rest NaN.  An empty
    request gives ``o = 0``, ``lse = -inf``."""
    qn, qp = to_f64(q_nope), to_f64(q_pe)
    B, H, R = qn.shape
    P = int(ckv_cache.shape[1])
    want = None
    if rows is not None:
        want = {}
        for b, h in rows:
            want.setdefault(int(b), set()).add(int(h))
    o = np.full((B, H, R), np.nan)
    lse = np.full((B, H), np.nan)
    for b in range(B):
        if want is not None and b not in want:
            continue
        toks = request_tokens(kv_indptr, kv_page_indices, kv_last_page_len, P, b)
        heads = range(H) if want is None else sorted(want[b])
        if not toks:
            for h in heads:
                o[b, h], lse[b, h] = 0.0, -math.inf
            continue
        pages = sorted({p for p, _ in toks})
        remap = {p: i for i, p in enumerate(pages)}
        import torch  # only to index the pages of a torch tensor
        sel = torch.as_tensor(pages, dtype=torch.long)
        ck = to_f64(ckv_cache[sel] if isinstance(ckv_cache, torch.Tensor) else np.asarray(ckv_cache)[pages])
        kp = to_f64(kpe_cache[sel] if isinstance(kpe_cache, torch.Tensor) else np.asarray(kpe_cache)[pages])
        pi = np.fromiter((remap[p] for p, _ in toks), dtype=np.int64, count=len(toks))
        si = np.fromiter((t for _, t in toks), dtype=np.int64, count=len(toks))
        c = ck[pi, si]  # [L, 512]
        r = kp[pi, si]  # [L, 64]
        for h in heads:
            s = sm_scale * (c @ qn[b, h] + r @ qp[b, h])
            m = float(np.max(s))
            ls = m + math.log(float(np.sum(np.exp(s - m))))
            o[b, h] = np.exp(s - ls) @ c
            lse[b, h] = ls
    return o, lse
