"""The allocation-free decode entry point (pkd_decode_noalloc) through the C ABI.

pkd_decode_noalloc serves callers that may not allocate device memory while
they run attention -- memory pooled up front by their own allocator, or owned
by a host runtime they are plugged into -- by using a scratch area built into
the library in place of a caller workspace.  Its output must match the fp64
oracle and the plan/run path within the parity tolerances, call after call,
even though every call reuses the same scratch bytes, and no call may leave a
device error bit set.

This file sorts last so that, in a run that stops at the first failure, every
other test has already run.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import _build
from paged_kv_decode_28_gb300 import api
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def _plan_run(b, idx):
    plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    out, lse = plan.run(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    return out, lse


def _noalloc(b, idx):
    out = torch.empty_like(b.q)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device=b.q.device)
    api.decode_noalloc(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, b.q, b.k_cache, b.v_cache, out, lse,
                       sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert api.noalloc_device_errors() == 0
    return out, lse


def _oracle(b):
    return orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices, b.kv_last_page_len,
                            sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale)


def test_noalloc_matches_oracle_and_plan_run_on_two_calls_in_a_row():
    first = wl.make_config(2, device="cuda", batch=16)
    second = wl.make_paged(seed=77, lengths=[0, 1, 15, 16, 17, 300, 4096, 0, 999, 64, 65, 2000],
                           num_qo_heads=64, num_kv_heads=8, page_size=16, device="cuda")
    for b in (first, second):
        idx = torch.from_numpy(b.kv_page_indices.copy()).cuda()
        got_o, got_l = _noalloc(b, idx)
        o_ref, l_ref = _oracle(b)
        assert_o_close(got_o, o_ref, what=f"{b.name} out vs oracle")
        assert_lse_close(got_l, l_ref, what=f"{b.name} lse vs oracle")
        ref_o, ref_l = _plan_run(b, idx)
        assert_o_close(got_o, ref_o.double().cpu().numpy(), what=f"{b.name} out vs plan/run")
        assert_lse_close(got_l, ref_l.double().cpu().numpy(), what=f"{b.name} lse vs plan/run")


def test_noalloc_fp8_pool_matches_oracle():
    b = wl.make_paged(seed=78, lengths=[1, 63, 64, 65, 700, 2049], num_qo_heads=32, num_kv_heads=4, page_size=64,
                      q_dtype="bf16", kv_dtype="e4m3", device="cuda")
    idx = torch.from_numpy(b.kv_page_indices.copy()).cuda()
    got_o, got_l = _noalloc(b, idx)
    o_ref, l_ref = _oracle(b)
    assert_o_close(got_o, o_ref, what="e4m3 out vs oracle")
    assert_lse_close(got_l, l_ref, what="e4m3 lse vs oracle")


def test_noalloc_out_of_range_page_is_flagged_then_cleared():
    b = wl.make_paged(seed=79, lengths=[40, 20], num_qo_heads=8, num_kv_heads=8, page_size=16, device="cuda")
    bad = b.kv_page_indices.copy()
    bad[1] = b.num_pages + 5  # a page id past the pool
    out = torch.empty_like(b.q)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device="cuda")
    api.decode_noalloc(b.kv_indptr, torch.from_numpy(bad).cuda(), b.kv_last_page_len, 16, b.q, b.k_cache, b.v_cache,
                       out, lse, sm_scale=b.sm_scale)
    assert api.noalloc_device_errors() == 1  # PKD_DEVERR_PAGE_INDEX
    # the next call starts from a clear error word
    _noalloc(b, torch.from_numpy(b.kv_page_indices.copy()).cuda())


def test_noalloc_batch_zero():
    q = torch.zeros(0, 32, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(0, 32, device="cuda")
    api.decode_noalloc(np.zeros(1, np.int32), torch.zeros(1, dtype=torch.int32, device="cuda"),
                       np.zeros(0, np.int32), 16, q, k, k, out, lse)
    torch.cuda.synchronize()
    assert api.noalloc_device_errors() == 0


def _accepts(batch, Hq=64, Hk=8):
    """Whether a call of `batch` empty requests fits the fixed scratch."""
    q = torch.zeros(batch, Hq, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, Hk, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(batch, Hq, device="cuda")
    try:
        api.decode_noalloc(np.zeros(batch + 1, np.int32), torch.zeros(1, dtype=torch.int32, device="cuda"),
                           np.zeros(batch, np.int32), 16, q, k, k, out, lse)
    except pkd.PkdError as e:
        assert e.status == 4 and "device scratch" in str(e), str(e)
        return False
    torch.cuda.synchronize()
    assert api.noalloc_device_errors() == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    return True


def test_noalloc_capacity_boundary():
    # the scratch is sized by batch x kv heads x group (not by lengths): find the
    # largest batch that fits with empty requests, then run real keys there
    lo, hi = 1, 4096
    assert _accepts(lo) and not _accepts(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if _accepts(mid):
            lo = mid
        else:
            hi = mid
    rng = np.random.default_rng(5)
    lengths = rng.integers(1, 80, size=lo).tolist()
    b = wl.make_paged(seed=80, lengths=lengths, num_qo_heads=64, num_kv_heads=8, page_size=16, device="cuda")
    idx = torch.from_numpy(b.kv_page_indices.copy()).cuda()
    got_o, got_l = _noalloc(b, idx)  # just under the limit
    o_ref, l_ref = _oracle(b)
    assert_o_close(got_o, o_ref, what=f"batch {lo} out vs oracle")
    assert_lse_close(got_l, l_ref, what=f"batch {lo} lse vs oracle")
    assert not _accepts(lo + 1)  # just over


def test_noalloc_refuses_a_capturing_stream():
    b = wl.make_paged(seed=81, lengths=[30], num_qo_heads=8, num_kv_heads=8, page_size=16, device="cuda")
    idx = torch.from_numpy(b.kv_page_indices.copy()).cuda()
    out = torch.zeros_like(b.q)
    lse = torch.empty(1, 8, device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    err = None
    with torch.cuda.graph(g, stream=s):
        out.add_(0)
        try:
            api.decode_noalloc(b.kv_indptr, idx, b.kv_last_page_len, 16, b.q, b.k_cache, b.v_cache, out, lse,
                               sm_scale=b.sm_scale)
        except pkd.PkdError as e:
            err = e
    assert err is not None and err.status == 2 and "captured" in str(err)
    # an eager call afterwards still works
    got_o, got_l = _noalloc(b, idx)
    o_ref, l_ref = _oracle(b)
    assert_o_close(got_o, o_ref)
    assert_lse_close(got_l, l_ref)
