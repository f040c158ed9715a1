"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
a library attention routine, closed forms, brute force on tiny inputs,
invariances the definition implies, and the deep-dive page's toy page table."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _contiguous_request(batch, b):
    """Request b's keys/values, built from the generator's own lengths (not the
    oracle's page walk): pages in table order, first kv_lens[b] tokens."""
    pages = batch.kv_page_indices[batch.kv_indptr[b]:batch.kv_indptr[b + 1]]
    L = int(batch.kv_lens[b])
    k = batch.k_cache[torch.as_tensor(pages, dtype=torch.long)].reshape(-1, batch.num_kv_heads, batch.head_dim)[:L]
    v = batch.v_cache[torch.as_tensor(pages, dtype=torch.long)].reshape(-1, batch.num_kv_heads, batch.head_dim)[:L]
    return k.to(torch.float64), v.to(torch.float64)


def _sdpa_reference(batch, k_scale=None, v_scale=None):
    """torch.nn.functional.scaled_dot_product_attention in fp64 on CPU, GQA by
    repeating kv heads, plus torch.logsumexp of the scaled scores."""
    g = batch.num_qo_heads // batch.num_kv_heads
    outs, lses = [], []
    for b in range(batch.batch):
        k, v = _contiguous_request(batch, b)
        if k_scale is not None:
            k = k * k_scale.to(torch.float64)[None, :, None]
            v = v * v_scale.to(torch.float64)[None, :, None]
        q = batch.q[b].to(torch.float64)  # [Hq, D]
        kk = k.repeat_interleave(g, dim=1).permute(1, 0, 2)  # [Hq, L, D]
        vv = v.repeat_interleave(g, dim=1).permute(1, 0, 2)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[:, None, :], kk, vv, scale=batch.sm_scale)[:, 0, :]
        s = torch.einsum("hd,hld->hl", q, kk) * batch.sm_scale
        outs.append(o.numpy())
        lses.append(torch.logsumexp(s, dim=-1).numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("P,Hq,Hk,kv", [(16, 8, 2, "bf16"), (4, 4, 4, "f16"), (64, 16, 2, "bf16"), (1, 6, 3, "f16")])
def test_oracle_matches_library_attention(P, Hq, Hk, kv):
    batch = wl.make_paged(seed=11, lengths=[1, P - 1 if P > 1 else 2, P, P + 1, 3 * P + 5, 97],
                          num_qo_heads=Hq, num_kv_heads=Hk, head_dim=32, page_size=P,
                          q_dtype=kv, kv_dtype=kv, pool_pages=200)
    o, lse = orc.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                              batch.kv_page_indices, batch.kv_last_page_len, sm_scale=batch.sm_scale)
    o_ref, lse_ref = _sdpa_reference(batch)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_oracle_fp8_scales_per_kv_head():
    batch = wl.make_paged(seed=12, lengths=[40, 129, 64], num_qo_heads=8, num_kv_heads=4,
                          head_dim=32, page_size=16, q_dtype="bf16", kv_dtype="e4m3", pool_pages=64)
    # make the heads' scales very different so a head mix-up cannot pass
    batch.k_scale = torch.tensor([0.5, 2.0, 0.125, 4.0])
    batch.v_scale = torch.tensor([3.0, 0.25, 1.0, 8.0])
    o, lse = orc.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                              batch.kv_page_indices, batch.kv_last_page_len, sm_scale=batch.sm_scale,
                              k_scale=batch.k_scale, v_scale=batch.v_scale)
    o_ref, lse_ref = _sdpa_reference(batch, batch.k_scale, batch.v_scale)
    # values reach a few thousand (codes up to 448 times scales up to 8)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_e4m3_known_codes():
    """OCP FP8 E4M3: 0x38 = 1, 0xB8 = -1, 0x7E = 448 (largest), 0x01 = 2^-9
    (smallest subnormal), 0x08 = 2^-6 (smallest normal)."""
    codes = torch.tensor([0x38, 0xB8, 0x7E, 0x01, 0x08], dtype=torch.uint8).view(torch.float8_e4m3fn)
    got = orc.to_f64(codes)
    np.testing.assert_array_equal(got, [1.0, -1.0, 448.0, 2.0 ** -9, 2.0 ** -6])


def test_single_key_is_exact():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal(16), rng.standard_normal((1, 16)), rng.standard_normal((1, 16))
    o, lse = orc.attend(q, k, v, 0.3)
    assert np.array_equal(o, v[0])
    assert lse == 0.3 * float(np.dot(k[0], q))


def test_two_keys_closed_form():
    """o = sigmoid(s0 - s1) v0 + sigmoid(s1 - s0) v1; lse = s0 + log1p(exp(s1 - s0))."""
    rng = np.random.default_rng(1)
    q, k, v = rng.standard_normal(8), rng.standard_normal((2, 8)), rng.standard_normal((2, 8))
    sc = 0.7
    s0, s1 = sc * float(k[0] @ q), sc * float(k[1] @ q)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))
    o_ref = sig(s0 - s1) * v[0] + sig(s1 - s0) * v[1]
    lse_ref = s0 + math.log1p(math.exp(s1 - s0))
    o, lse = orc.attend(q, k, v, sc)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-14)
    assert abs(lse - lse_ref) < 1e-14


def test_constant_values_give_that_value():
    rng = np.random.default_rng(2)
    L, D = 300, 16
    q, k = rng.standard_normal(D) * 3, rng.standard_normal((L, D))
    row = rng.standard_normal(D)
    o, _ = orc.attend(q, k, np.tile(row, (L, 1)), 1.0)
    np.testing.assert_allclose(o, row, rtol=0, atol=1e-13)


def test_zero_query_is_mean_and_log_length():
    rng = np.random.default_rng(3)
    L, D = 123, 16
    k, v = rng.standard_normal((L, D)), rng.standard_normal((L, D))
    o, lse = orc.attend(np.zeros(D), k, v, 0.5)
    np.testing.assert_allclose(o, v.mean(axis=0), rtol=0, atol=1e-14)
    assert abs(lse - math.log(L)) < 1e-13


def test_lse_bounds():
    rng = np.random.default_rng(4)
    for L in (1, 2, 17, 500):
        q, k, v = rng.standard_normal(16), rng.standard_normal((L, 16)), rng.standard_normal((L, 16))
        _, lse = orc.attend(q, k, v, 2.0)
        smax = float(np.max(2.0 * (k @ q)))
        assert smax - 1e-12 <= lse <= smax + math.log(L) + 1e-12


def test_empty_request_state():
    batch = wl.make_paged(seed=5, lengths=[0, 5, 0], num_qo_heads=2, num_kv_heads=1, head_dim=8,
                          page_size=4, q_dtype="f16", kv_dtype="f16", pool_pages=4)
    o, lse = orc.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                              batch.kv_page_indices, batch.kv_last_page_len)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(o[2] == 0) and np.all(np.isneginf(lse[2]))
    assert np.all(np.isfinite(lse[1]))


def test_page_relabelling_invariance():
    batch = wl.make_paged(seed=6, lengths=[50, 7, 33], num_qo_heads=4, num_kv_heads=2, head_dim=16,
                          page_size=8, kv_dtype="bf16", pool_pages=40)
    args = dict(sm_scale=batch.sm_scale)
    o1, l1 = orc.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                              batch.kv_page_indices, batch.kv_last_page_len, **args)
    perm = np.random.default_rng(7).permutation(batch.num_pages)  # old page p -> new slot perm[p]
    inv = np.argsort(perm)
    k2 = batch.k_cache[torch.as_tensor(inv)]
    v2 = batch.v_cache[torch.as_tensor(inv)]
    idx2 = perm[batch.kv_page_indices].astype(np.int32)
    o2, l2 = orc.paged_decode(batch.q, k2, v2, batch.kv_indptr, idx2, batch.kv_last_page_len, **args)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_page_size_repacking_invariance():
    """The same key sequence stored with page sizes 1, 16 and 64 gives one result."""
    rng = np.random.default_rng(8)
    lengths = [1, 15, 16, 17, 130]
    Hk, D = 2, 16
    seqs_k = [rng.standard_normal((L, Hk, D)) for L in lengths]
    seqs_v = [rng.standard_normal((L, Hk, D)) for L in lengths]
    q = torch.as_tensor(rng.standard_normal((len(lengths), 4, D)))
    results = []
    for P in (1, 16, 64):
        n = [(L + P - 1) // P for L in lengths]
        order = rng.permutation(sum(n) + 3)
        indptr, idx, last = wl.lengths_to_page_table(lengths, P, order)
        kc = np.zeros((len(order), P, Hk, D))
        vc = np.zeros((len(order), P, Hk, D))
        for b, L in enumerate(lengths):
            for t in range(L):
                page = idx[indptr[b] + t // P]
                kc[page, t % P] = seqs_k[b][t]
                vc[page, t % P] = seqs_v[b][t]
        results.append(orc.paged_decode(q, kc, vc, indptr, idx, last, sm_scale=0.25))
    for o, l in results[1:]:
        np.testing.assert_allclose(o, results[0][0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, results[0][1], rtol=0, atol=1e-12)


@pytest.mark.parametrize("split", [1, 16, 37, 99, 127])
def test_merge_of_disjoint_parts_is_attention_of_union(split):
    rng = np.random.default_rng(9 + split)
    L, D = 128, 32
    q, k, v = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    o, s = orc.attend(q, k, v, 0.2)
    oa, sa = orc.attend(q, k[:split], v[:split], 0.2)
    ob, sb = orc.attend(q, k[split:], v[split:], 0.2)
    om, sm = orc.merge_state(oa, np.float64(sa), ob, np.float64(sb))
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-13)
    assert abs(float(sm) - s) < 1e-13
    # commutativity
    om2, sm2 = orc.merge_state(ob, np.float64(sb), oa, np.float64(sa))
    np.testing.assert_allclose(om2, om, rtol=0, atol=1e-15)
    assert abs(float(sm2) - float(sm)) < 1e-15


def test_merge_with_empty_state():
    rng = np.random.default_rng(10)
    v = rng.standard_normal((3, 4, 8))
    s = rng.standard_normal((3, 4))
    empty_v, empty_s = np.zeros_like(v), np.full_like(s, -np.inf)
    for a, b in (((v, s), (empty_v, empty_s)), ((empty_v, empty_s), (v, s))):
        vm, sm = orc.merge_state(a[0], a[1], b[0], b[1])
        np.testing.assert_array_equal(vm, v)
        np.testing.assert_array_equal(sm, s)
    vm, sm = orc.merge_state(empty_v, empty_s, empty_v, empty_s)
    assert np.all(vm == 0) and np.all(np.isneginf(sm))


def test_merge_states_equals_attention_over_all_parts():
    rng = np.random.default_rng(11)
    L, D, k_parts = 200, 16, 5
    q, K, V = rng.standard_normal(D), rng.standard_normal((L, D)), rng.standard_normal((L, D))
    cuts = [0, 1, 50, 51, 130, 200]
    vs, ss = [], []
    for i in range(k_parts):
        o, s = orc.attend(q, K[cuts[i]:cuts[i + 1]], V[cuts[i]:cuts[i + 1]], 0.3)
        vs.append(o)
        ss.append(s)
    v = np.asarray(vs)[None, :, None, :]
    s = np.asarray(ss)[None, :, None]
    vm, sm = orc.merge_states(v, s)
    o_all, s_all = orc.attend(q, K, V, 0.3)
    np.testing.assert_allclose(vm[0, 0], o_all, rtol=0, atol=1e-13)
    assert abs(sm[0, 0] - s_all) < 1e-13


def test_cascade_equals_plain_decode_over_prefix_then_suffix():
    batch = wl.make_paged(seed=13, lengths=[5, 40, 16, 1], num_qo_heads=8, num_kv_heads=2,
                          head_dim=16, page_size=8, kv_dtype="bf16", prefix_len=72)
    o, s = orc.cascade_decode(batch.q, batch.k_cache, batch.v_cache, batch.prefix_page_indices,
                              batch.prefix_last_page_len, batch.kv_indptr, batch.kv_page_indices,
                              batch.kv_last_page_len, sm_scale=batch.sm_scale)
    plain = wl.cascade_as_plain(batch)
    o2, s2 = orc.paged_decode(plain.q, plain.k_cache, plain.v_cache, plain.kv_indptr,
                              plain.kv_page_indices, plain.kv_last_page_len, sm_scale=batch.sm_scale)
    np.testing.assert_allclose(o, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(s, s2, rtol=0, atol=1e-12)


def test_single_decode_quickstart_shapes_match_paged():
    """Contiguous [L, Hk, D] K/V equals the same data as an identity-ordered page table."""
    gen = torch.Generator().manual_seed(14)
    q = torch.randn(32, 128, generator=gen).half()
    k = torch.randn(2048, 32, 128, generator=gen).half()
    v = torch.randn(2048, 32, 128, generator=gen).half()
    o1, l1 = orc.single_decode(q, k, v)
    P = 16
    indptr = np.array([0, 128], np.int32)
    idx = np.arange(128, dtype=np.int32)
    last = np.array([16], np.int32)
    o2, l2 = orc.paged_decode(q[None], k.view(128, P, 32, 128), v.view(128, P, 32, 128), indptr, idx, last)
    np.testing.assert_allclose(o1, o2[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2[0], rtol=0, atol=1e-13)


def test_deep_dive_toy_page_table():
    g = json.load(open(os.path.join(GOLDEN, "p4_toy_page_table.json")))
    lists = g["page_lists"]
    P = g["page_size"]
    lengths = [len(x) * P for x in lists]  # all pages full (see the fixture's reading)
    order = np.concatenate([np.asarray(x) for x in lists])
    indptr, idx, last = wl.lengths_to_page_table(lengths, P, order)
    assert indptr.tolist() == g["expected_kv_indptr"]
    assert idx.tolist() == g["expected_kv_page_indices"]
    assert last.tolist() == g["expected_kv_last_page_len"]
    for b, pages in enumerate(lists):
        toks = orc.request_tokens(indptr, idx, last, P, b)
        assert len(toks) == g["expected_kv_len"][b]
        assert toks == [(p, t) for p in pages for t in range(P)]
    # the combined [pages, 2, P, H, D] pool read through K/V views equals separate pools
    H, D = 4, 16  # the snippet's 32 x 128 heads shrunk to keep the test fast
    pool = torch.randn(11, 2, P, H, D, generator=torch.Generator().manual_seed(15), dtype=torch.float64)
    q = torch.randn(3, H, D, generator=torch.Generator().manual_seed(16), dtype=torch.float64)
    o1, l1 = orc.paged_decode(q, pool[:, 0], pool[:, 1], indptr, idx, last)
    o2, l2 = orc.paged_decode(q, pool[:, 0].clone(), pool[:, 1].clone(), indptr, idx, last)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
