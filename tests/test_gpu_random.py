"""Seeded random geometries through the GPU paths, against the fp64 oracle:
batch size, group size, kv heads, page size (any size the plan accepts), dtype
pair and the length mix (empty requests, a few keys, a page and a key either
side of it, thousands of keys) drawn per seed, so that the combinations the
hand-picked cases miss are covered too.  Large cases compare sampled rows."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close, gpu_paged_decode, sample_rows

pytestmark = pytest.mark.gpu

DTYPES = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "e4m3"), ("f16", "e4m3")]


def _page_size(rng):
    # any of 1..64, or a multiple of 64
    return int(rng.integers(1, 65)) if rng.random() < 0.7 else int(64 * rng.integers(1, 5))


def _lengths(rng, B, P, longest):
    kinds = rng.integers(0, 5, size=B)
    out = []
    for k in kinds:
        if k == 0:
            out.append(0)
        elif k == 1:
            out.append(int(rng.integers(1, 4)))
        elif k == 2:
            out.append(int(max(1, P + rng.integers(-1, 2))))
        else:
            out.append(int(rng.integers(1, longest + 1)))
    return out


def _rows(b, n, seed):
    if b.batch * b.num_qo_heads <= 2 * n:
        return None
    return sample_rows(b, n, seed=seed)


@pytest.mark.parametrize("seed", range(24))
def test_random_decode(seed):
    rng = np.random.default_rng(5000 + seed)
    qd, kvd = DTYPES[seed % 4]
    g = int(rng.integers(1, 9))
    Hk = int(rng.choice([1, 2, 4, 8]))
    P = _page_size(rng)
    B = int(rng.integers(1, 41))
    lengths = _lengths(rng, B, P, 2500)
    b = wl.make_paged(seed=5100 + seed, lengths=lengths, num_qo_heads=g * Hk, num_kv_heads=Hk, page_size=P,
                      q_dtype=qd, kv_dtype=kvd, device="cuda")
    out, lse, _ = gpu_paged_decode(b)
    rows = _rows(b, 64, seed)
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices, b.kv_last_page_len,
                                    sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("seed", range(12))
def test_random_cascade(seed):
    rng = np.random.default_rng(6000 + seed)
    qd, kvd = DTYPES[seed % 4]
    g = int(rng.integers(1, 9))
    Hk = int(rng.choice([1, 2, 4]))
    P = _page_size(rng)
    B = int(rng.integers(1, 301))
    prefix_len = int(rng.integers(1, 3001))
    lengths = _lengths(rng, B, P, 300)
    b = wl.make_paged(seed=6100 + seed, lengths=lengths, num_qo_heads=g * Hk, num_kv_heads=Hk, page_size=P,
                      q_dtype=qd, kv_dtype=kvd, prefix_len=prefix_len, device="cuda")
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_page_indices)).cuda()
    pre = torch.from_numpy(np.ascontiguousarray(b.prefix_page_indices)).cuda()
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    out, lse = plan.cascade_decode(pre, b.prefix_last_page_len, b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale,
                                   k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    rows = _rows(b, 64, seed)
    o_ref, l_ref = orc.cascade_decode(b.q, b.k_cache, b.v_cache, b.prefix_page_indices, b.prefix_last_page_len,
                                      b.kv_indptr, b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale,
                                      k_scale=b.k_scale, v_scale=b.v_scale, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("seed", range(8))
def test_random_tree(seed):
    rng = np.random.default_rng(7000 + seed)
    dt = "bf16" if seed % 2 == 0 else "f16"
    g = int(rng.choice([1, 2, 4, 8]))  # the tile kernel's group sizes divide 128
    Hk = int(rng.choice([1, 2, 4]))
    P = int(rng.choice([1, 2, 8, 16, 32, 64, 128, 192]))
    B = int(rng.integers(1, 200))
    levels = []
    for l in range(int(rng.integers(1, 4))):
        n_nodes = 1 if l == 0 else int(rng.integers(1, min(B, 6) + 1))
        cuts = np.sort(rng.choice(np.arange(1, B), size=n_nodes - 1, replace=False)) if n_nodes > 1 else []
        counts = np.diff(np.concatenate([[0], cuts, [B]])).astype(int).tolist()
        toks = rng.integers(0, 1500, size=n_nodes).tolist()
        levels.append((counts, toks))
    lengths = _lengths(rng, B, P, 200)
    b = wl.make_tree(seed=7100 + seed, levels=levels, lengths=lengths, num_qo_heads=g * Hk, num_kv_heads=Hk,
                     page_size=P, q_dtype=dt, kv_dtype=dt, device="cuda")
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_page_indices)).cuda()
    dev_levels = [(ri, ki, torch.as_tensor(np.asarray(pg, dtype=np.int32)).cuda(), last)
                  for ri, ki, pg, last in b.levels]
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    plan.plan_tree(dev_levels)
    out, lse = plan.tree_decode(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    rows = _rows(b, 64, seed)
    o_ref, l_ref = orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels, b.kv_indptr,
                                                 b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale,
                                                 rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("seed", range(8))
def test_random_decode_hnd(seed):
    """The same draws on HND pages ([pages, Hk, P, D]), against the oracle on
    the NHD copy."""
    from tests.test_gpu_hnd import to_hnd

    rng = np.random.default_rng(5500 + seed)
    qd, kvd = DTYPES[seed % 4]
    g = int(rng.integers(1, 9))
    Hk = int(rng.choice([1, 2, 4, 8]))
    P = _page_size(rng)
    B = int(rng.integers(1, 41))
    lengths = _lengths(rng, B, P, 2000)
    b = wl.make_paged(seed=5600 + seed, lengths=lengths, num_qo_heads=g * Hk, num_kv_heads=Hk, page_size=P,
                      q_dtype=qd, kv_dtype=kvd, device="cuda")
    idx = torch.as_tensor(np.asarray(b.kv_page_indices, np.int32)).cuda()
    plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads, kv_layout="HND")
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    out, lse = plan.run(b.q, to_hnd(b.k_cache), to_hnd(b.v_cache), sm_scale=b.sm_scale, k_scale=b.k_scale,
                        v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    rows = _rows(b, 64, seed)
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices, b.kv_last_page_len,
                                    sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("seed", range(10))
def test_random_prefill(seed):
    rng = np.random.default_rng(8000 + seed)
    dt = "bf16" if seed % 2 == 0 else "f16"
    g = int(rng.choice([1, 2, 4, 8]))
    Hk = int(rng.choice([1, 2, 4]))
    P = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 128, 192]))
    B = int(rng.integers(1, 13))
    causal = bool(rng.integers(0, 2))
    kv_lens = rng.integers(1, 2001, size=B)
    q_lens = [int(rng.integers(0, min(k, 600) + 1)) for k in kv_lens]
    b = wl.make_prefill(seed=8100 + seed, q_lens=q_lens, kv_lens=kv_lens.tolist(), num_qo_heads=g * Hk,
                        num_kv_heads=Hk, page_size=P, q_dtype=dt, kv_dtype=dt, device="cuda")
    plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads)
    plan.plan_prefill(b.qo_indptr, b.kv_indptr, torch.as_tensor(np.asarray(b.kv_page_indices, np.int32)).cuda(),
                      b.kv_last_page_len, b.page_size, causal=causal, q_dtype=b.q.dtype)
    out, lse = plan.prefill(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    n_rows = int(sum(q_lens)) * b.num_qo_heads
    rows = None
    if n_rows > 4096:
        r = np.random.default_rng(seed)
        rows = sorted({(int(t), int(h)) for t, h in zip(r.integers(0, int(sum(q_lens)), 96),
                                                        r.integers(0, b.num_qo_heads, 96))})
    o_ref, l_ref = orc.paged_prefill(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                     b.kv_last_page_len, causal=causal, sm_scale=b.sm_scale, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("seed", range(8))
def test_random_mla(seed):
    from oracle import mla as orc_mla

    rng = np.random.default_rng(9000 + seed)
    H = int(rng.integers(1, 129))
    P = int(rng.choice([1, 2, 4, 8, 16, 32, 64, 96, 128]))
    B = int(rng.integers(1, 25))
    lengths = _lengths(rng, B, P, 3000)
    b = wl.make_mla(seed=9100 + seed, lengths=lengths, num_heads=H, page_size=P, device="cuda")
    idx = torch.as_tensor(np.asarray(b.kv_page_indices, np.int32)).cuda()
    out, lse, ws = pkd.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, idx, b.kv_last_page_len,
                                  sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert int(ws[:4].view(torch.int32).item()) == 0
    rows = None
    if B * H > 256:
        r = np.random.default_rng(seed)
        rows = sorted({(int(q), int(h)) for q, h in zip(r.integers(0, B, 64), r.integers(0, H, 64))})
    o_ref, l_ref = orc_mla.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, b.kv_page_indices,
                                      b.kv_last_page_len, sm_scale=b.sm_scale, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)
