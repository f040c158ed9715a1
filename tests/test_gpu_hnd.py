"""GPU parity of HND pools ([num_pages, Hk, page_size, 128] pages, one head's
keys contiguous) for every path that reads or writes the cache: batched decode,
cascade decode, the allocation-free entry point and the KV append.  The oracle
attends NHD pools, so each case builds the NHD pool, checks the HND run
against the oracle on it, and also checks that the HND run returns exactly
what the NHD run returns (the kernels read the same rows into the same
shared-memory tiles whatever the layout)."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from oracle import kv_append as ka
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close, gpu_paged_decode

pytestmark = pytest.mark.gpu

DTYPES = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "e4m3"), ("f16", "e4m3")]


def to_hnd(cache: torch.Tensor) -> torch.Tensor:
    """An NHD pool [N, P, Hk, D] as a contiguous HND pool [N, Hk, P, D] (a byte copy)."""
    return cache.view(torch.uint8).permute(0, 2, 1, 3).contiguous().view(cache.dtype)


def from_hnd(cache: torch.Tensor) -> torch.Tensor:
    return cache.view(torch.uint8).permute(0, 2, 1, 3).contiguous().view(cache.dtype)


def _cuda_i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _hnd_decode(b, kh, vh):
    idx = _cuda_i32(b.kv_page_indices)
    plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads, kv_layout="HND")
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=kh.dtype)
    out, lse = plan.run(b.q, kh, vh, sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    return out, lse


@pytest.mark.parametrize("qd,kvd", DTYPES)
@pytest.mark.parametrize("P", [1, 16, 48, 64, 128])
@pytest.mark.parametrize("g", [1, 8])
def test_hnd_decode_matches_oracle_and_nhd(qd, kvd, P, g):
    lengths = [1, max(P - 1, 1), P, P + 1, 63, 64, 65, 200, 0, 777]
    b = wl.make_paged(seed=900 + P + g, lengths=lengths, num_qo_heads=2 * g, num_kv_heads=2, page_size=P,
                      q_dtype=qd, kv_dtype=kvd, device="cuda")
    out_n, lse_n, _ = gpu_paged_decode(b)
    out_h, lse_h = _hnd_decode(b, to_hnd(b.k_cache), to_hnd(b.v_cache))
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                    b.kv_last_page_len, sm_scale=b.sm_scale, k_scale=b.k_scale,
                                    v_scale=b.v_scale)
    assert_o_close(out_h, o_ref)
    assert_lse_close(lse_h, l_ref)
    assert torch.equal(out_h, out_n) and torch.equal(lse_h, lse_n)


def test_hnd_workload_geometry():
    """The batch-64 GQA workload cut to 16 requests, HND pool."""
    b = wl.make_config(2, device="cuda", batch=16)
    out_h, lse_h = _hnd_decode(b, to_hnd(b.k_cache), to_hnd(b.v_cache))
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                    b.kv_last_page_len, sm_scale=b.sm_scale)
    assert_o_close(out_h, o_ref)
    assert_lse_close(lse_h, l_ref)


def test_hnd_interleaved_pool():
    """One [pages, 2, Hk, P, D] pool, K and V read through views with a 2-page stride."""
    b = wl.make_paged(seed=930, lengths=[64, 32, 80, 300], num_qo_heads=32, num_kv_heads=8, page_size=16,
                      pool_pages=64, device="cuda")
    pool = torch.stack([to_hnd(b.k_cache), to_hnd(b.v_cache)], dim=1).contiguous()
    kh, vh = pool[:, 0], pool[:, 1]
    assert kh.stride(0) == 2 * 8 * 16 * 128
    out_h, lse_h = _hnd_decode(b, kh, vh)
    out_n, lse_n, _ = gpu_paged_decode(b)
    assert torch.equal(out_h, out_n) and torch.equal(lse_h, lse_n)
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                    b.kv_last_page_len, sm_scale=b.sm_scale)
    assert_o_close(out_h, o_ref)


@pytest.mark.parametrize("P", [1, 16, 64, 128])
def test_hnd_cascade_matches_oracle_and_nhd(P):
    b = wl.make_paged(seed=940 + P, lengths=[33, 0, 200, 1, 65], num_qo_heads=16, num_kv_heads=4, page_size=P,
                      prefix_len=3 * 128 + 7, device="cuda")
    idx = _cuda_i32(b.kv_page_indices)
    pre = _cuda_i32(b.prefix_page_indices)
    res = {}
    for layout in ("NHD", "HND"):
        kc, vc = (b.k_cache, b.v_cache) if layout == "NHD" else (to_hnd(b.k_cache), to_hnd(b.v_cache))
        plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16, kv_layout=layout)
        plan.plan(b.kv_indptr, idx, b.kv_last_page_len, P, q_dtype=b.q.dtype, kv_dtype=kc.dtype)
        res[layout] = plan.cascade_decode(pre, b.prefix_last_page_len, b.q, kc, vc, sm_scale=b.sm_scale)
        torch.cuda.synchronize()
        assert plan.check_device_errors() == 0
    o_ref, l_ref = orc.cascade_decode(b.q, b.k_cache, b.v_cache, b.prefix_page_indices, b.prefix_last_page_len,
                                      b.kv_indptr, b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale)
    assert_o_close(res["HND"][0], o_ref)
    assert_lse_close(res["HND"][1], l_ref)
    assert torch.equal(res["HND"][0], res["NHD"][0]) and torch.equal(res["HND"][1], res["NHD"][1])


@pytest.mark.parametrize("kvd", ["bf16", "e4m3"])
def test_hnd_noalloc_equals_nhd(kvd):
    b = wl.make_paged(seed=950, lengths=[5, 300, 0, 64, 1000], num_qo_heads=16, num_kv_heads=4, page_size=16,
                      kv_dtype=kvd, device="cuda")
    idx = _cuda_i32(b.kv_page_indices)
    outs = {}
    for layout in ("NHD", "HND"):
        kc, vc = (b.k_cache, b.v_cache) if layout == "NHD" else (to_hnd(b.k_cache), to_hnd(b.v_cache))
        out = torch.empty_like(b.q)
        lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device="cuda")
        pkd.decode_noalloc(b.kv_indptr, idx, b.kv_last_page_len, 16, b.q, kc, vc, out, lse, sm_scale=b.sm_scale,
                           k_scale=b.k_scale, v_scale=b.v_scale, kv_layout=layout)
        torch.cuda.synchronize()
        outs[layout] = (out, lse)
    assert torch.equal(outs["HND"][0], outs["NHD"][0]) and torch.equal(outs["HND"][1], outs["NHD"][1])
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                    b.kv_last_page_len, sm_scale=b.sm_scale, k_scale=b.k_scale,
                                    v_scale=b.v_scale)
    assert_o_close(outs["HND"][0], o_ref)
    assert_lse_close(outs["HND"][1], l_ref)


@pytest.mark.parametrize("kvd,newd", [("bf16", torch.bfloat16), ("f16", torch.float16), ("e4m3", torch.bfloat16)])
@pytest.mark.parametrize("P", [1, 16, 64])
def test_hnd_append_matches_oracle_bit_for_bit(kvd, newd, P):
    lens = np.array([0, 5, 15, 16, 63, 64, 200])
    b = wl.make_paged(seed=960 + P, lengths=(lens + 1).tolist(), num_qo_heads=16, num_kv_heads=4, page_size=P,
                      kv_dtype=kvd, q_dtype="bf16", device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(9)
    n, Hk = len(lens), b.num_kv_heads
    k_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(newd)
    v_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(newd)
    kr, vr, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, np.arange(n), lens, b.kv_indptr,
                                   b.kv_page_indices, P, b.k_scale, b.v_scale)
    assert skipped == 0
    kh, vh = to_hnd(b.k_cache), to_hnd(b.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(k_new, v_new, _cuda_i32(np.arange(n)), _cuda_i32(lens), _cuda_i32(b.kv_indptr),
                  _cuda_i32(b.kv_page_indices), kh, vh, k_scale=b.k_scale, v_scale=b.v_scale, err=err,
                  kv_layout="HND")
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(from_hnd(kh).cpu().view(torch.uint8), kr.view(torch.uint8))
    assert torch.equal(from_hnd(vh).cpu().view(torch.uint8), vr.view(torch.uint8))


def test_hnd_arguments_are_checked():
    b = wl.make_paged(seed=970, lengths=[16], num_qo_heads=4, num_kv_heads=2, page_size=16, device="cuda")
    with pytest.raises(ValueError):
        pkd.Plan(1, 4, 2, kv_layout="NDH")
    plan = pkd.Plan(1, 4, 2, kv_layout="HND")
    plan.plan(b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, 16)
    with pytest.raises(ValueError):  # an NHD-shaped pool (16 slots, 2 heads) is not [N, Hk, P, D]
        plan.run(b.q, b.k_cache, b.v_cache)
