"""Pins of the oracle's prefix-tree cascade and prefill / append attention
against facts the oracle does not compute itself: a library attention routine
over keys gathered straight from the generator's tables (not the oracle's page
walk), invariances the definitions imply, and reductions to the pinned decode
oracle."""
import numpy as np
import pytest
import torch

from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl


def _pages_keys(batch, pages, n_tokens):
    """K and V rows of the first n_tokens slots of the given pages, in order."""
    idx = torch.as_tensor(np.asarray(pages, np.int64), dtype=torch.long)
    k = batch.k_cache[idx].reshape(-1, batch.num_kv_heads, batch.head_dim)[:n_tokens]
    v = batch.v_cache[idx].reshape(-1, batch.num_kv_heads, batch.head_dim)[:n_tokens]
    return k.to(torch.float64), v.to(torch.float64)


def _library_attention(q, k, v, scale, g, causal_offset=None):
    """torch SDPA in fp64 for q [n, Hq, D] over k, v [L, Hk, D] (GQA by
    repeating kv heads) and torch.logsumexp of the scaled scores.  With
    causal_offset c, query row i sees keys 0 .. c + i only (each row is its
    own library call over the truncated keys)."""
    kk = k.repeat_interleave(g, dim=1).permute(1, 0, 2)  # [Hq, L, D]
    vv = v.repeat_interleave(g, dim=1).permute(1, 0, 2)
    outs, lses = [], []
    for i in range(q.shape[0]):
        n = kk.shape[1] if causal_offset is None else causal_offset + i + 1
        qi = q[i].to(torch.float64)
        o = torch.nn.functional.scaled_dot_product_attention(qi[:, None, :], kk[:, :n], vv[:, :n], scale=scale)[:, 0]
        s = torch.einsum("hd,hld->hl", qi, kk[:, :n]) * scale
        outs.append(o.numpy())
        lses.append(torch.logsumexp(s, dim=-1).numpy())
    return np.stack(outs), np.stack(lses)


def _tree():
    return wl.make_tree(seed=71, levels=[([6], [37]), ([2, 3, 1], [16, 0, 21]), ([1, 1, 1, 2, 1], [3, 1, 0, 9, 4])],
                        lengths=[0, 5, 17, 1, 33, 2], num_qo_heads=8, num_kv_heads=2, page_size=4)


def test_tree_equals_library_attention_over_the_concatenated_keys():
    b = _tree()
    o, lse = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels, b.kv_indptr, b.kv_page_indices,
                                           b.kv_last_page_len, sm_scale=b.sm_scale)
    g = b.num_qo_heads // b.num_kv_heads
    for r in range(b.batch):
        ks, vs = [], []
        for req_indptr, ip, idx, last in b.levels:
            n = int(np.searchsorted(req_indptr, r, side="right") - 1)
            pages = idx[ip[n]:ip[n + 1]]
            toks = (len(pages) - 1) * b.page_size + int(last[n]) if len(pages) else 0
            k, v = _pages_keys(b, pages, toks)
            ks.append(k)
            vs.append(v)
        k, v = _pages_keys(b, b.kv_page_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]], int(b.kv_lens[r]))
        k, v = torch.cat(ks + [k]), torch.cat(vs + [v])
        o_ref, l_ref = _library_attention(b.q[r:r + 1], k, v, b.sm_scale, g)
        assert np.allclose(o[r], o_ref[0], rtol=0, atol=1e-12)
        assert np.allclose(lse[r], l_ref[0], rtol=0, atol=1e-12)


def test_tree_is_invariant_to_level_order():
    b = _tree()
    a = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels, b.kv_indptr, b.kv_page_indices,
                                      b.kv_last_page_len, sm_scale=b.sm_scale)
    r = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels[::-1], b.kv_indptr, b.kv_page_indices,
                                      b.kv_last_page_len, sm_scale=b.sm_scale)
    assert np.allclose(a[0], r[0], rtol=0, atol=1e-12) and np.allclose(a[1], r[1], rtol=0, atol=1e-12)


def test_tree_level_of_empty_nodes_is_the_identity():
    b = _tree()
    empty = (np.array([0, 4, 6], np.int32), np.array([0, 0, 0], np.int32), np.zeros(0, np.int32),
             np.zeros(2, np.int32))
    a = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels, b.kv_indptr, b.kv_page_indices,
                                      b.kv_last_page_len, sm_scale=b.sm_scale)
    e = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels[:1] + [empty] + b.levels[1:],
                                      b.kv_indptr, b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale)
    assert np.array_equal(a[0], e[0]) and np.array_equal(a[1], e[1])


def test_tree_rejects_nodes_that_do_not_partition_the_batch():
    b = _tree()
    bad = (np.array([0, 4], np.int32), np.array([0, 1], np.int32), np.array([0], np.int32), np.array([2], np.int32))
    with pytest.raises(ValueError):
        orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, [bad], b.kv_indptr, b.kv_page_indices,
                                      b.kv_last_page_len)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_equals_library_attention(causal):
    q_lens, kv_lens = [3, 0, 5, 1, 16], [10, 4, 5, 1, 40]
    b = wl.make_prefill(seed=72, q_lens=q_lens, kv_lens=kv_lens, num_qo_heads=8, num_kv_heads=2, page_size=4)
    o, lse = orc.paged_prefill(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                               b.kv_last_page_len, causal=causal, sm_scale=b.sm_scale)
    g = 4
    for r in range(len(q_lens)):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        if q1 == q0:
            continue
        k, v = _pages_keys(b, b.kv_page_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]], kv_lens[r])
        off = kv_lens[r] - q_lens[r] if causal else None
        o_ref, l_ref = _library_attention(b.q[q0:q1], k, v, b.sm_scale, g, off)
        assert np.allclose(o[q0:q1], o_ref, rtol=0, atol=1e-12)
        assert np.allclose(lse[q0:q1], l_ref, rtol=0, atol=1e-12)


def test_causal_prefill_of_a_whole_sequence_is_library_causal_attention():
    """q_len == kv_len: the bottom-right causal mask is the usual lower-triangular one."""
    L = 23
    b = wl.make_prefill(seed=73, q_lens=[L], kv_lens=[L], num_qo_heads=4, num_kv_heads=4, page_size=8)
    o, _ = orc.paged_prefill(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                             b.kv_last_page_len, causal=True, sm_scale=b.sm_scale)
    k, v = _pages_keys(b, b.kv_page_indices, L)
    ref = torch.nn.functional.scaled_dot_product_attention(
        b.q.to(torch.float64).permute(1, 0, 2), k.permute(1, 0, 2), v.permute(1, 0, 2), is_causal=True,
        scale=b.sm_scale).permute(1, 0, 2)
    assert np.allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_last_prefill_token_is_decode_over_all_keys():
    q_lens, kv_lens = [4, 1, 7], [9, 30, 7]
    b = wl.make_prefill(seed=74, q_lens=q_lens, kv_lens=kv_lens, num_qo_heads=6, num_kv_heads=3, page_size=4)
    o, lse = orc.paged_prefill(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                               b.kv_last_page_len, causal=True, sm_scale=b.sm_scale)
    last = b.qo_indptr[1:] - 1
    od, ld = orc.paged_decode(b.q[torch.as_tensor(last, dtype=torch.long)], b.k_cache, b.v_cache, b.kv_indptr,
                              b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale)
    assert np.array_equal(o[last], od) and np.array_equal(lse[last], ld)
