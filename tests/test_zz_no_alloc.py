"""The allocation-free decode entry point (pkd_decode_noalloc) against the
regular plan/run path, through the C ABI.

pkd_decode_noalloc serves callers that may not allocate device memory while
they run attention -- memory pooled up front by their own allocator, or owned
by a host runtime they are plugged into -- by using a scratch area built into
the library in place of a caller workspace.  Its output must match the
plan/run path within the parity tolerances, call after call, even though every
call reuses the same scratch bytes.

This file sorts last so that, in a run that stops at the first failure, every
other test has already run.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from paged_kv_decode_28_gb300 import _build
from paged_kv_decode_28_gb300 import api
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def _plan_run(b, idx):
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads)
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
    return out, lse


def test_noalloc_matches_plan_run_on_two_calls_in_a_row():
    first = wl.make_config(2, device="cuda", batch=16)
    second = wl.make_paged(seed=77, lengths=[0, 1, 15, 16, 17, 300, 4096, 0, 999, 64, 65, 2000],
                           num_qo_heads=64, num_kv_heads=8, page_size=16, device="cuda")
    for b in (first, second):
        idx = torch.from_numpy(b.kv_page_indices.copy()).cuda()
        ref_o, ref_l = _plan_run(b, idx)
        got_o, got_l = _noalloc(b, idx)
        assert_o_close(got_o, ref_o.double().cpu().numpy(), what=f"{b.name} out")
        assert_lse_close(got_l, ref_l.double().cpu().numpy(), what=f"{b.name} lse")


def test_noalloc_rejects_work_beyond_its_scratch():
    B, Hq, Hk = 4096, 8, 8
    q = torch.zeros(B, Hq, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 16, Hk, 128, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, device="cuda")
    indptr = np.zeros(B + 1, np.int32)
    last = np.zeros(B, np.int32)
    with pytest.raises(pkd.PkdError) as e:
        api.decode_noalloc(indptr, idx, last, 16, q, k, k, out, lse)
    assert e.value.status == 4
    assert "scratch" in str(e.value)
