"""GPU parity of cascade (shared-prefix) decode: the tcgen05 prefix kernel,
the all-partial suffix decode and the merge pass, against the fp64 oracle's
merge_state(attn(prefix), attn(suffix)); plus edge cases (one-key prefix,
partial query tiles, empty suffixes, no prefix)."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close, sample_rows

pytestmark = pytest.mark.gpu


def _gpu_cascade(b, plan=None):
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_page_indices)).cuda()
    pre = torch.from_numpy(np.ascontiguousarray(b.prefix_page_indices)).cuda() if b.prefix_page_indices is not None \
        else torch.zeros(0, dtype=torch.int32, device="cuda")
    if plan is None:
        plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    out, lse = plan.cascade_decode(pre, b.prefix_last_page_len, b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale,
                                   k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    return out, lse


def _oracle(b, rows=None):
    pre = b.prefix_page_indices if b.prefix_page_indices is not None else np.zeros(0, np.int32)
    return orc.cascade_decode(b.q, b.k_cache, b.v_cache, pre, b.prefix_last_page_len, b.kv_indptr,
                              b.kv_page_indices, b.kv_last_page_len, sm_scale=b.sm_scale, k_scale=b.k_scale,
                              v_scale=b.v_scale, rows=rows)


@pytest.mark.parametrize("prefix_len", [1, 15, 63, 64, 65, 127, 128, 129, 191, 1000])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_cascade_small(prefix_len, g):
    b = wl.make_paged(seed=200 + prefix_len + g, lengths=[0, 1, 17, 300, 64, 5, 129], num_qo_heads=2 * g,
                      num_kv_heads=2, page_size=16, prefix_len=prefix_len, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("prefix_len", [1, 2, 3])
def test_cascade_few_prefix_keys_many_requests(prefix_len):
    """A prefix of 1-3 keys and suffixes of 0-2 keys for many requests: the
    prefix state is a sum of 1-3 value rows, so the weights' precision in the
    tensor-core P V product shows at full size."""
    rng = np.random.default_rng(62 + prefix_len)
    lengths = rng.integers(0, 3, size=300).tolist()
    b = wl.make_paged(seed=620 + prefix_len, lengths=lengths, num_qo_heads=16, num_kv_heads=2, page_size=16,
                      prefix_len=prefix_len, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("prefix_len", [1, 2, 63, 64, 65, 128, 129, 1000])
@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
def test_cascade_e4m3_pool(prefix_len, q_dtype):
    """E4M3 K/V with per-kv-head scales: the prefix codes are widened exactly
    to q's type before the tensor-core products."""
    b = wl.make_paged(seed=700 + prefix_len, lengths=[0, 1, 17, 300, 64, 5, 129], num_qo_heads=16,
                      num_kv_heads=4, page_size=16, q_dtype=q_dtype, kv_dtype="e4m3", prefix_len=prefix_len,
                      device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("prefix_len", [1, 3])
def test_cascade_e4m3_few_prefix_keys_many_requests(prefix_len):
    rng = np.random.default_rng(72 + prefix_len)
    lengths = rng.integers(0, 3, size=300).tolist()
    b = wl.make_paged(seed=720 + prefix_len, lengths=lengths, num_qo_heads=16, num_kv_heads=2, page_size=64,
                      q_dtype="bf16", kv_dtype="e4m3", prefix_len=prefix_len, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_e4m3_long_context_sampled():
    """The long-context fp8 geometry (64 / 8 heads, page 64) with a shared
    prefix of 8192 keys and 160 requests, sampled rows."""
    rng = np.random.default_rng(73)
    lengths = rng.integers(64, 2048, size=160).tolist()
    b = wl.make_paged(seed=730, lengths=lengths, num_qo_heads=64, num_kv_heads=8, page_size=64,
                      q_dtype="bf16", kv_dtype="e4m3", prefix_len=8192, device="cuda")
    out, lse = _gpu_cascade(b)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = sample_rows(b, 40, seed=73)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("g", [3, 5, 6, 7])
@pytest.mark.parametrize("prefix_len", [1, 200, 1000])
def test_cascade_odd_groups(g, prefix_len):
    """Group sizes that do not divide 128: a CTA holds floor(128 / g) requests
    and its last rows stay empty; batches leave the last pair half empty."""
    rng = np.random.default_rng(g * 10 + prefix_len)
    B = 2 * (128 // g) + 5  # three CTA row tiles: the second pair's odd CTA is past the batch
    lens = rng.integers(0, 300, size=B)
    b = wl.make_paged(seed=740 + g + prefix_len, lengths=lens, num_qo_heads=2 * g, num_kv_heads=2, page_size=16,
                      prefix_len=prefix_len, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("prefix_len", [1, 47, 48, 49, 130, 1000])
@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_cascade_page_48(prefix_len, kv_dtype):
    """A page size that is neither a divisor of the 128-key tile nor a multiple
    of 64: boxes of gcd(48, 64) = 16 keys, tiles straddling pages."""
    b = wl.make_paged(seed=760 + prefix_len, lengths=[0, 1, 47, 48, 49, 500], num_qo_heads=32, num_kv_heads=8,
                      page_size=48, q_dtype="bf16", kv_dtype=kv_dtype, prefix_len=prefix_len, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("P", [1, 4, 64, 128])
def test_cascade_page_sizes(P):
    b = wl.make_paged(seed=300 + P, lengths=[33, 0, 200, 1], num_qo_heads=16, num_kv_heads=4, page_size=P,
                      prefix_len=3 * 128 + 7, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("B", [1, 31, 33, 70, 100, 200])
def test_cascade_partial_query_tiles(B):
    """B * g rows not a multiple of the 128-row tile (and odd tile counts, where
    a CTA's second query tile lies past the batch): padded rows must not leak."""
    rng = np.random.default_rng(B)
    lens = rng.integers(0, 400, size=B)
    b = wl.make_paged(seed=400 + B, lengths=lens, num_qo_heads=32, num_kv_heads=8, page_size=16,
                      prefix_len=2048, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_growing_scores():
    """Prefix keys whose norm grows along the prefix, so the running max rises
    by more than the lazy-rescale threshold many times (O rescaled in TMEM)."""
    b = wl.make_paged(seed=502, lengths=[3, 90, 0, 400], num_qo_heads=16, num_kv_heads=2, page_size=16,
                      prefix_len=1000, device="cuda")
    for pos, pid in enumerate(b.prefix_page_indices.tolist()):
        b.k_cache[pid] *= 1.0 + 0.25 * pos
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_f16():
    b = wl.make_paged(seed=500, lengths=[10, 200, 0, 77], num_qo_heads=16, num_kv_heads=2, page_size=16,
                      q_dtype="f16", kv_dtype="f16", prefix_len=777, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_without_prefix_is_plain_decode():
    b = wl.make_paged(seed=501, lengths=[10, 200, 0, 77], num_qo_heads=16, num_kv_heads=2, page_size=16,
                      device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                    b.kv_last_page_len, sm_scale=b.sm_scale)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_equals_decode_over_prefix_then_suffix():
    b = wl.make_config(4, device="cuda", batch=24)
    out, lse = _gpu_cascade(b)
    plain = wl.cascade_as_plain(b)
    idx = torch.from_numpy(plain.kv_page_indices).cuda()
    plan = pkd.Plan(plain.batch, plain.num_qo_heads, plain.num_kv_heads)
    plan.plan(plain.kv_indptr, idx, plain.kv_last_page_len, plain.page_size)
    o2, l2 = plan.run(plain.q, plain.k_cache, plain.v_cache, sm_scale=plain.sm_scale)
    torch.cuda.synchronize()
    assert_o_close(out, o2.double().cpu().numpy())
    assert_lse_close(lse, l2.double().cpu().numpy())


def test_cascade_workload_full_size_sampled():
    b = wl.make_config(4, device="cuda")
    out, lse = _gpu_cascade(b)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = sample_rows(b, 40, seed=4)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_cascade_is_deterministic_and_replans():
    b = wl.make_config(4, device="cuda", batch=40)
    plan = pkd.Plan(64, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    o1, l1 = _gpu_cascade(b, plan)
    o2, l2 = _gpu_cascade(b, plan)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_cascade_back_to_back_without_sync():
    """Cascade steps of two alternating batches with no host synchronization:
    the prefix kernel of one step runs beside the tail of its decode grid and
    must leave the previous step's merge inputs alone."""
    batches = [wl.make_config(4, device="cuda", batch=24), wl.make_config(4, device="cuda", batch=40)]
    plan = pkd.Plan(64, 32, 8, max_prefix_splits=16)
    refs = [_gpu_cascade(b, plan) for b in batches]
    refs = [(o.clone(), l.clone()) for o, l in refs]
    outs = []
    for i in range(6):
        b = batches[i % 2]
        idx = torch.from_numpy(np.ascontiguousarray(b.kv_page_indices)).cuda()
        pre = torch.from_numpy(np.ascontiguousarray(b.prefix_page_indices)).cuda()
        plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size)
        outs.append(plan.cascade_decode(pre, b.prefix_last_page_len, b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale))
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    for i, (o, l) in enumerate(outs):
        ro, rl = refs[i % 2]
        assert torch.equal(o, ro) and torch.equal(l, rl), f"step {i} differs from the isolated run"


@pytest.mark.parametrize("P", [1, 3, 7, 23, 33, 63])
@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
def test_cascade_e4m3_odd_page_sizes(P, q_dtype):
    """Odd page sizes give single-key copy boxes in the prefix kernel: its e4m3
    V rows (64 codes) then land 128 bytes apart, each copy's destination
    128-byte aligned."""
    rng = np.random.default_rng(990 + P)
    lengths = rng.integers(0, 70, size=37).tolist()
    b = wl.make_paged(seed=995 + P, lengths=lengths, num_qo_heads=12, num_kv_heads=4, page_size=P, q_dtype=q_dtype,
                      kv_dtype="e4m3", prefix_len=300 + P, device="cuda")
    out, lse = _gpu_cascade(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)
