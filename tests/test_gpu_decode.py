"""GPU parity of batched paged decode (plan + run through the C ABI) against the
fp64 oracle: small cases spanning several chunks and ragged tails, edge
lengths, every supported dtype pair and page size, the standard workloads at
reduced and full size (sampled rows), determinism and device error flags."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import (assert_lse_close, assert_o_close, gpu_paged_decode, sample_rows,
                          to_device)

pytestmark = pytest.mark.gpu

DTYPES = [("bf16", "bf16"), ("f16", "f16"), ("bf16", "e4m3"), ("f16", "e4m3")]


def _oracle(b, rows=None):
    return orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices, b.kv_last_page_len,
                            sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale, rows=rows)


@pytest.mark.parametrize("qd,kvd", DTYPES)
@pytest.mark.parametrize("P", [1, 16, 48, 64, 128])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_small_batches_edge_lengths(qd, kvd, P, g):
    lengths = [1, max(P - 1, 1), P, P + 1, 63, 64, 65, 200, 0, 777]
    b = wl.make_paged(seed=100 + P + g, lengths=lengths, num_qo_heads=2 * g, num_kv_heads=2,
                      page_size=P, q_dtype=qd, kv_dtype=kvd, device="cuda")
    out, lse, _ = gpu_paged_decode(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("qd,kvd", DTYPES)
def test_few_keys_many_requests(qd, kvd):
    """Requests of 1-3 keys: with so few keys the output is a sum of 1-3 value
    rows whose weights are not averaged out, so an error in the weights passed
    to the P V product (e.g. rounding P to the 16-bit type) shows at full size,
    and cancellations make |o| small against the absolute tolerance."""
    rng = np.random.default_rng(61)
    lengths = rng.integers(1, 4, size=400).tolist()
    for P, g in ((1, 8), (16, 4), (64, 1)):
        b = wl.make_paged(seed=610 + P + g, lengths=lengths, num_qo_heads=2 * g, num_kv_heads=2, page_size=P,
                          q_dtype=qd, kv_dtype=kvd, device="cuda")
        out, lse, _ = gpu_paged_decode(b)
        o_ref, l_ref = _oracle(b)
        assert_o_close(out, o_ref)
        assert_lse_close(lse, l_ref)


def test_batch_of_one_and_all_empty():
    b = wl.make_paged(seed=7, lengths=[37], num_qo_heads=8, num_kv_heads=1, page_size=16, device="cuda")
    out, lse, _ = gpu_paged_decode(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)
    e = wl.make_paged(seed=8, lengths=[0, 0, 0], num_qo_heads=4, num_kv_heads=4, page_size=16,
                      pool_pages=4, device="cuda")
    out, lse, _ = gpu_paged_decode(e)
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


def test_interleaved_kv_pool():
    """The deep dive's combined [pages, 2, P, H, D] pool, read through K/V views."""
    b = wl.make_paged(seed=9, lengths=[64, 32, 80, 300], num_qo_heads=32, num_kv_heads=8, page_size=16,
                      pool_layout="interleaved", pool_pages=64, device="cuda")
    assert b.k_cache.stride(0) == 2 * 16 * 8 * 128
    out, lse, _ = gpu_paged_decode(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("idx,batch", [(1, None), (2, 8), (3, 12), (4, 16), (5, 2)])
def test_standard_workloads_reduced(idx, batch):
    b = wl.make_config(idx, device="cuda", batch=batch)
    if idx == 4:
        b = wl.cascade_as_plain(b)  # cascade workload as plain paged decode over prefix ++ suffix
    out, lse, _ = gpu_paged_decode(b)
    rows = None if idx != 5 else sample_rows(b, 24)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("idx", [1, 2, 3, 5])
def test_standard_workloads_full_size_sampled(idx):
    b = wl.make_config(idx, device="cuda")
    out, lse, _ = gpu_paged_decode(b)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = sample_rows(b, 16 if idx == 5 else 48, seed=idx)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_runs_are_bit_identical():
    b = wl.make_config(3, device="cuda", batch=24)
    out1, lse1, plan = gpu_paged_decode(b)
    out2, lse2 = plan.run(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_single_decode_quickstart():
    """single_decode_with_kv_cache shapes: q [32, 128], K/V [2048, 32, 128] fp16."""
    g = torch.Generator(device="cuda").manual_seed(1)
    q = torch.randn(32, 128, device="cuda", generator=g).half()
    k = torch.randn(2048, 32, 128, device="cuda", generator=g).half()
    v = torch.randn(2048, 32, 128, device="cuda", generator=g).half()
    o, lse = pkd.single_decode(q, k, v)
    o_ref, l_ref = orc.single_decode(q, k, v)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, l_ref)


def test_single_decode_into_given_outputs():
    """out / lse given: written in place, two calls in a row with different
    inputs; wrong output shapes are refused."""
    g = torch.Generator(device="cuda").manual_seed(2)
    out = torch.full((32, 128), float("nan"), device="cuda").half()
    lse = torch.full((32,), float("nan"), device="cuda")
    for L in (300, 77):
        q = torch.randn(32, 128, device="cuda", generator=g).half()
        k = torch.randn(L, 8, 128, device="cuda", generator=g).half()
        v = torch.randn(L, 8, 128, device="cuda", generator=g).half()
        o, s = pkd.single_decode(q, k, v, out=out, lse=lse)
        assert o.data_ptr() == out.data_ptr() and s.data_ptr() == lse.data_ptr()
        o_ref, l_ref = orc.single_decode(q, k, v)
        assert_o_close(out, o_ref)
        assert_lse_close(lse, l_ref)
    with pytest.raises(ValueError):
        pkd.single_decode(q, k, v, out=torch.empty(16, 128, device="cuda").half())
    with pytest.raises(ValueError):
        pkd.single_decode(q, k, v, lse=torch.empty(32, device="cuda").half())


@pytest.mark.parametrize("L", [0, 1, 63, 64, 65, 100, 1000])
def test_single_decode_lengths_gqa(L):
    g = torch.Generator(device="cuda").manual_seed(L)
    q = torch.randn(16, 128, device="cuda", generator=g).bfloat16()
    k = torch.randn(L, 4, 128, device="cuda", generator=g).bfloat16()
    v = torch.randn(L, 4, 128, device="cuda", generator=g).bfloat16()
    o, lse = pkd.single_decode(q, k, v, sm_scale=0.05)
    if L == 0:
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
        return
    o_ref, l_ref = orc.single_decode(q, k, v, sm_scale=0.05)
    assert_o_close(o, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("L", [1, 65, 2048])
def test_single_decode_captured_in_a_graph(L):
    """The schedule of single-request decode travels in its upload kernel's
    parameters, so the call captures into a CUDA graph; replays after the
    inputs change in place follow the new values."""
    g = torch.Generator(device="cuda").manual_seed(300 + L)
    q = torch.randn(32, 128, device="cuda", generator=g).half()
    k = torch.randn(L, 8, 128, device="cuda", generator=g).half()
    v = torch.randn(L, 8, 128, device="cuda", generator=g).half()
    ws = torch.empty(pkd.workspace_bytes(1, 32, 8, 128, pkd.num_ctas(0), 0), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkd.single_decode(q, k, v, workspace=ws)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        o, lse = pkd.single_decode(q, k, v, workspace=ws)
    for rep in range(3):
        q.copy_(torch.randn(32, 128, device="cuda", generator=g).half())
        k.copy_(torch.randn(L, 8, 128, device="cuda", generator=g).half())
        v.copy_(torch.randn(L, 8, 128, device="cuda", generator=g).half())
        graph.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = orc.single_decode(q, k, v)
        assert_o_close(o, o_ref)
        assert_lse_close(lse, l_ref)


def test_out_of_range_page_index_sets_flag():
    """A page id past the pool is read as page 0 and flagged; nothing faults."""
    b = wl.make_paged(seed=10, lengths=[40, 40], num_qo_heads=8, num_kv_heads=2, page_size=16,
                      pool_pages=8, device="cuda")
    b.kv_page_indices = b.kv_page_indices.copy()
    b.kv_page_indices[1] = b.num_pages + 5
    out, lse, plan = gpu_paged_decode(b, check_errors=False)
    flags = plan.check_device_errors()
    assert flags & pkd.api.DEVERR_PAGE_INDEX
    assert plan.check_device_errors() == 0  # cleared


def test_bad_arguments_raise():
    b = wl.make_paged(seed=11, lengths=[40], num_qo_heads=8, num_kv_heads=2, page_size=16, device="cuda")
    plan = pkd.Plan(1, 8, 2)
    idx = torch.from_numpy(b.kv_page_indices).cuda()
    with pytest.raises(pkd.PkdError):
        plan.run(b.q, b.k_cache, b.v_cache)  # run before plan
    with pytest.raises(pkd.PkdError):
        plan.plan([0, 3, 2], idx, [16, 16], 16)  # decreasing indptr
    with pytest.raises(pkd.PkdError):
        plan.plan(b.kv_indptr, idx, b.kv_last_page_len, 16, q_dtype=torch.float16, kv_dtype=torch.bfloat16)
    with pytest.raises(pkd.PkdError):
        big = pkd.Plan(1, 8, 2)
        big.plan([0, 1, 2], idx, [16, 16], 16)  # batch above max_batch


@pytest.mark.parametrize("qd,kvd", [("bf16", "bf16"), ("bf16", "e4m3")])
@pytest.mark.parametrize("g", [2, 3, 5, 6, 7])
def test_group_sizes_not_powers_of_two(qd, kvd, g):
    """GQA groups of 2..7 qo heads per kv head (padded to the 16 MMA rows)."""
    b = wl.make_paged(seed=600 + g, lengths=[1, 65, 300, 0, 1500], num_qo_heads=3 * g, num_kv_heads=3,
                      page_size=16, q_dtype=qd, kv_dtype=kvd, device="cuda")
    out, lse, _ = gpu_paged_decode(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_one_request_of_a_million_keys():
    """One (request, kv head) row cut into one item per CTA: the merge folds
    hundreds of partial states, more than one warp-wide batch of them."""
    b = wl.make_paged(seed=610, lengths=[1 << 20], num_qo_heads=8, num_kv_heads=1, page_size=16, device="cuda")
    plan = pkd.Plan(1, 8, 1)
    sched = pkd.plan_host(b.kv_indptr, b.kv_last_page_len, 1, 16, plan.num_ctas)
    assert sched["row_item_count"][0] > 32  # more states than one warp-wide batch
    out, lse, plan = gpu_paged_decode(b, plan)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_run_without_lse_output():
    """d_lse = NULL is allowed: out must equal the run that also writes lse."""
    b = wl.make_paged(seed=620, lengths=[5, 700, 2000, 64], num_qo_heads=16, num_kv_heads=4, page_size=16,
                      device="cuda")
    out, lse, plan = gpu_paged_decode(b)
    out2 = torch.empty_like(out)
    N, P, Hk, D = b.k_cache.shape
    stride = b.k_cache.stride(0)
    st = pkd.api.lib().pkd_run(plan._h, b.q.data_ptr(), b.k_cache.data_ptr(), b.v_cache.data_ptr(), N, stride,
                               None, None, float(b.sm_scale), out2.data_ptr(), None,
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    assert torch.equal(out, out2)


def test_stalled_pipeline_times_out_flags_and_recovers():
    """A decode pipeline whose producer issues nothing (host-set test hook):
    every wait runs out after its ~2 s limit, the kernel returns with
    PKD_DEVERR_WAIT_TIMEOUT set, and the context stays usable for a normal run."""
    import time
    b = wl.make_paged(seed=630, lengths=[40, 300, 1000], num_qo_heads=8, num_kv_heads=2, page_size=16,
                      device="cuda")
    out, lse, plan = gpu_paged_decode(b)
    plan.set_debug(1)
    t0 = time.perf_counter()
    plan.run(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    flags = plan.check_device_errors()
    assert flags & pkd.api.DEVERR_WAIT_TIMEOUT, f"flags {flags:#x}"
    assert 1.0 < waited < 30.0, f"the stalled kernel returned after {waited:.2f} s"
    plan.set_debug(0)
    out2, lse2 = plan.run(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    o_ref, l_ref = _oracle(b)
    assert_o_close(out2, o_ref)
    assert_lse_close(lse2, l_ref)
