"""Pins of the MLA decode oracle (oracle/mla.py) against facts it does not
compute itself: library attention over the latent and rotary rows gathered
straight from the generator's tables, and the absorption identity the pages
describe (attending the latent cache with the key up-projection folded into
the query equals decompressing K and V per head and attending them)."""
import numpy as np
import pytest
import torch

from oracle import mla
from paged_kv_decode_28_gb300 import workloads as wl


def _rows(b, r):
    """Request r's latent and rotary rows from the generator's own lengths."""
    pages = torch.as_tensor(np.asarray(b.kv_page_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]], np.int64))
    L = int(b.kv_lens[r])
    c = b.ckv_cache[pages].reshape(-1, 512)[:L].to(torch.float64)
    k = b.kpe_cache[pages].reshape(-1, 64)[:L].to(torch.float64)
    return c, k


@pytest.mark.parametrize("P", [1, 16])
def test_mla_equals_library_attention(P):
    b = wl.make_mla(seed=81, lengths=[1, 17, 40, 0, 33], num_heads=8, page_size=P)
    o, lse = mla.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, b.kv_page_indices,
                            b.kv_last_page_len, sm_scale=b.sm_scale)
    for r in range(b.batch):
        c, k = _rows(b, r)
        if c.shape[0] == 0:
            assert np.all(o[r] == 0) and np.all(np.isneginf(lse[r]))
            continue
        q = torch.cat([b.q_nope[r], b.q_pe[r]], dim=-1).to(torch.float64)  # [H, 576]
        keys = torch.cat([c, k], dim=-1)  # [L, 576]
        ref = torch.nn.functional.scaled_dot_product_attention(q[:, None, :], keys[None], c[None],
                                                               scale=b.sm_scale)[:, 0]
        s = torch.logsumexp(q @ keys.T * b.sm_scale, dim=-1)
        assert np.allclose(o[r], ref.numpy(), rtol=0, atol=1e-12)
        assert np.allclose(lse[r], s.numpy(), rtol=0, atol=1e-12)


def test_absorbed_latent_attention_equals_decompressed_attention():
    """Per head h, random up-projections W_UK[h], W_UV[h] (512 x 128): standard
    attention of q_full = [q_h (128), q_pe] over K = [ckv W_UK[h], kpe] and
    V = ckv W_UV[h] equals the latent output times W_UV[h] when the kernel's
    query is q_nope = W_UK[h] q_h."""
    H = 4
    b = wl.make_mla(seed=82, lengths=[29, 64], num_heads=H, page_size=16)
    g = torch.Generator().manual_seed(5)
    w_uk = torch.randn(H, 512, 128, generator=g, dtype=torch.float64) / 8
    w_uv = torch.randn(H, 512, 128, generator=g, dtype=torch.float64) / 8
    q_full = torch.randn(b.batch, H, 128, generator=g, dtype=torch.float64)
    q_nope = torch.einsum("hrd,bhd->bhr", w_uk, q_full)  # the absorbed query, float64
    o, _ = mla.mla_decode(q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, b.kv_page_indices,
                          b.kv_last_page_len, sm_scale=b.sm_scale)
    for r in range(b.batch):
        c, k = _rows(b, r)
        for h in range(H):
            keys = torch.cat([c @ w_uk[h], k], dim=-1)  # decompressed per-head keys [L, 192]
            vals = c @ w_uv[h]  # [L, 128]
            q = torch.cat([q_full[r, h], b.q_pe[r, h].to(torch.float64)])
            ref = torch.nn.functional.scaled_dot_product_attention(q[None, None], keys[None], vals[None],
                                                                   scale=b.sm_scale)[0, 0]
            got = torch.as_tensor(o[r, h]) @ w_uv[h]
            assert torch.allclose(got, ref, rtol=0, atol=1e-10)
