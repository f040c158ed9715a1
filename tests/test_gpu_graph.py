"""CUDA-graph friendliness: run() captured once keeps its launch shape, and a
re-plan of new lengths followed by a replay (the mode the benchmark times)
matches the fp64 oracle and equals an eager run bit for bit; the same for a
captured cascade step."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def test_replan_then_replay_matches_eager():
    B, Hq, Hk, P = 16, 32, 8, 16
    pool = wl.make_paged(seed=30, lengths=[4096] * B, num_qo_heads=Hq, num_kv_heads=Hk, page_size=P,
                         device="cuda")
    plan = pkd.Plan(B, Hq, Hk)
    q = pool.q.clone()
    out = torch.empty_like(q)
    lse = torch.empty(B, Hq, device="cuda")
    rng = np.random.default_rng(0)

    def table(lens):
        n = (lens + P - 1) // P
        indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
        return indptr, last

    idx = torch.from_numpy(rng.permutation(pool.num_pages).astype(np.int32)).cuda()
    lens0 = rng.integers(1, 4096, size=B)
    indptr, last = table(lens0)
    plan.plan(indptr, idx, last, P)
    plan.run(q, pool.k_cache, pool.v_cache, out=out, lse=lse)  # warm-up outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            plan.run(q, pool.k_cache, pool.v_cache, out=out, lse=lse, stream=s)
    for trial in range(3):
        lens = rng.integers(0, 4096, size=B)
        indptr, last = table(lens)
        plan.plan(indptr, idx, last, P)
        graph.replay()
        torch.cuda.synchronize()
        assert plan.check_device_errors() == 0
        o_ref, l_ref = orc.paged_decode(q, pool.k_cache, pool.v_cache, indptr, idx.cpu().numpy(), last,
                                        sm_scale=pool.sm_scale)
        assert_o_close(out, o_ref, what=f"replay {trial} out")
        assert_lse_close(lse, l_ref, what=f"replay {trial} lse")
        eager = pkd.Plan(B, Hq, Hk)
        eager.plan(indptr, idx, last, P)
        o2, l2 = eager.run(q, pool.k_cache, pool.v_cache)
        torch.cuda.synchronize()
        assert torch.equal(out, o2), trial
        assert torch.equal(lse, l2), trial


def test_back_to_back_replans_without_sync():
    """plan/run pairs of alternating batches with no host synchronization: each
    run's upload may start while the previous step's merge drains and must not
    overwrite the schedule that merge reads, and plan must not overwrite a
    staged schedule before its upload has read it."""
    B, Hq, Hk, P = 12, 32, 8, 16
    pool = wl.make_paged(seed=31, lengths=[3000] * B, num_qo_heads=Hq, num_kv_heads=Hk, page_size=P,
                         device="cuda")
    rng = np.random.default_rng(1)
    idx = torch.from_numpy(rng.permutation(pool.num_pages).astype(np.int32)).cuda()

    def table(lens):
        n = (lens + P - 1) // P
        indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
        return indptr, last

    tables = [table(rng.integers(1, 3000, size=B)), table(rng.integers(0, 600, size=B))]
    plan = pkd.Plan(B, Hq, Hk)
    ref = []
    for indptr, last in tables:  # each batch alone, synchronized
        plan.plan(indptr, idx, last, P)
        o, l = plan.run(pool.q, pool.k_cache, pool.v_cache)
        torch.cuda.synchronize()
        o_ref, l_ref = orc.paged_decode(pool.q, pool.k_cache, pool.v_cache, indptr, idx.cpu().numpy(), last,
                                        sm_scale=pool.sm_scale)
        assert_o_close(o, o_ref)
        assert_lse_close(l, l_ref)
        ref.append((o.clone(), l.clone()))
    outs = [(torch.empty_like(pool.q), torch.empty(B, Hq, device="cuda")) for _ in range(8)]
    for i, (o, l) in enumerate(outs):
        indptr, last = tables[i % 2]
        plan.plan(indptr, idx, last, P)
        plan.run(pool.q, pool.k_cache, pool.v_cache, out=o, lse=l)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    for i, (o, l) in enumerate(outs):
        ro, rl = ref[i % 2]
        assert torch.equal(o, ro), f"step {i}: output differs from the isolated run"
        assert torch.equal(l, rl), f"step {i}: lse differs from the isolated run"


@pytest.mark.parametrize("kv_dtype", ["bf16"])
def test_cascade_replan_then_replay_matches_oracle(kv_dtype):
    """A cascade step (upload, suffix decode, prefix kernel, merge) captured
    once, replayed after re-plans of new suffix lengths, against the oracle's
    merge_state(attn(prefix), attn(suffix))."""
    B, Hq, Hk, P = 40, 32, 8, 16
    pool = wl.make_paged(seed=32, lengths=[512] * B, num_qo_heads=Hq, num_kv_heads=Hk, page_size=P,
                         prefix_len=1000, q_dtype="bf16", kv_dtype=kv_dtype, device="cuda")
    rng = np.random.default_rng(2)
    own = pool.kv_page_indices.copy()  # the suffix pages (32 per request), re-cut per trial
    idx = torch.from_numpy(own).cuda()
    pre = torch.from_numpy(pool.prefix_page_indices.copy()).cuda()
    plan = pkd.Plan(B, Hq, Hk, max_prefix_splits=16)
    out = torch.empty_like(pool.q)
    lse = torch.empty(B, Hq, device="cuda")
    kw = dict(sm_scale=pool.sm_scale, k_scale=pool.k_scale, v_scale=pool.v_scale, out=out, lse=lse)

    def table(lens):
        # request r keeps its first ceil(lens[r] / P) pages of the original 32
        n = (lens + P - 1) // P
        indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        pages = np.concatenate([own[32 * r:32 * r + n[r]] for r in range(B)]).astype(np.int32)
        last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
        return indptr, pages, last

    indptr, pages, last = table(rng.integers(0, 513, size=B))
    idx.copy_(torch.from_numpy(np.pad(pages, (0, len(own) - len(pages)))))
    plan.plan(indptr, idx, last, P, q_dtype=pool.q.dtype, kv_dtype=pool.k_cache.dtype)
    plan.cascade_decode(pre, pool.prefix_last_page_len, pool.q, pool.k_cache, pool.v_cache, **kw)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            plan.cascade_decode(pre, pool.prefix_last_page_len, pool.q, pool.k_cache, pool.v_cache, stream=s, **kw)
    for trial in range(3):
        indptr, pages, last = table(rng.integers(0, 513, size=B))
        idx.copy_(torch.from_numpy(np.pad(pages, (0, len(own) - len(pages)))))
        plan.plan(indptr, idx, last, P, q_dtype=pool.q.dtype, kv_dtype=pool.k_cache.dtype)
        graph.replay()
        torch.cuda.synchronize()
        assert plan.check_device_errors() == 0
        o_ref, l_ref = orc.cascade_decode(pool.q, pool.k_cache, pool.v_cache, pool.prefix_page_indices,
                                          pool.prefix_last_page_len, indptr, pages, last, sm_scale=pool.sm_scale,
                                          k_scale=pool.k_scale, v_scale=pool.v_scale)
        assert_o_close(out, o_ref, what=f"cascade replay {trial} out")
        assert_lse_close(lse, l_ref, what=f"cascade replay {trial} lse")


def test_cascade_back_to_back_without_sync():
    """Cascade steps of alternating suffix tables with no host synchronization:
    the prefix grid of a step must not overwrite the prefix pieces the previous
    step's merge still reads, and the suffix decode behind it must read its own
    step's schedule; every step equals its isolated run bit for bit."""
    B, Hq, Hk, P = 40, 32, 8, 16
    pool = wl.make_paged(seed=33, lengths=[512] * B, num_qo_heads=Hq, num_kv_heads=Hk, page_size=P,
                         prefix_len=1000, q_dtype="bf16", kv_dtype="bf16", device="cuda")
    rng = np.random.default_rng(3)
    own = pool.kv_page_indices.copy()
    pre = torch.from_numpy(pool.prefix_page_indices.copy()).cuda()
    plan = pkd.Plan(B, Hq, Hk, max_prefix_splits=16)

    def table(lens):
        n = (lens + P - 1) // P
        indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        pages = np.concatenate([own[32 * r:32 * r + n[r]] for r in range(B)]).astype(np.int32)
        last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
        return indptr, torch.from_numpy(np.ascontiguousarray(pages)).cuda(), last

    tables = [table(rng.integers(1, 513, size=B)), table(rng.integers(0, 65, size=B))]
    kw = dict(sm_scale=pool.sm_scale)
    ref = []
    for indptr, pages, last in tables:  # each alone, synchronized, against the oracle
        plan.plan(indptr, pages, last, P, q_dtype=pool.q.dtype, kv_dtype=pool.k_cache.dtype)
        o, l = plan.cascade_decode(pre, pool.prefix_last_page_len, pool.q, pool.k_cache, pool.v_cache, **kw)
        torch.cuda.synchronize()
        o_ref, l_ref = orc.cascade_decode(pool.q, pool.k_cache, pool.v_cache, pool.prefix_page_indices,
                                          pool.prefix_last_page_len, indptr, pages.cpu().numpy(), last,
                                          sm_scale=pool.sm_scale)
        assert_o_close(o, o_ref)
        assert_lse_close(l, l_ref)
        ref.append((o.clone(), l.clone()))
    outs = [(torch.empty_like(pool.q), torch.empty(B, Hq, device="cuda")) for _ in range(8)]
    for i, (o, l) in enumerate(outs):
        indptr, pages, last = tables[i % 2]
        plan.plan(indptr, pages, last, P, q_dtype=pool.q.dtype, kv_dtype=pool.k_cache.dtype)
        plan.cascade_decode(pre, pool.prefix_last_page_len, pool.q, pool.k_cache, pool.v_cache, out=o, lse=l, **kw)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    for i, (o, l) in enumerate(outs):
        ro, rl = ref[i % 2]
        assert torch.equal(o, ro), f"step {i}: output differs from the isolated run"
        assert torch.equal(l, rl), f"step {i}: lse differs from the isolated run"
