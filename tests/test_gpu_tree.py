"""GPU parity of prefix-tree (multi-level cascade) decode: the tile-attention
kernel over every shared level's nodes, the requests' own decode and the merge
of all parts, against the oracle's per-level states merged with merge_state;
plus empty nodes and levels, page sizes, group sizes, HND pools, a
serving-size tree with sampled rows, graph replay across re-plans and
argument checks."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close, sample_rows

pytestmark = pytest.mark.gpu


def _cuda_i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _dev_levels(b):
    return [(ri, ki, _cuda_i32(idx), last) for ri, ki, idx, last in b.levels]


def _gpu_tree(b, plan=None, layout="NHD", kc=None, vc=None):
    if plan is None:
        plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16, kv_layout=layout)
    plan.plan(b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype,
              kv_dtype=b.k_cache.dtype)
    plan.plan_tree(_dev_levels(b))
    out, lse = plan.tree_decode(b.q, b.k_cache if kc is None else kc, b.v_cache if vc is None else vc,
                                sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    return out, lse


def _oracle(b, rows=None):
    return orc.multilevel_cascade_decode(b.q, b.k_cache, b.v_cache, b.levels, b.kv_indptr, b.kv_page_indices,
                                         b.kv_last_page_len, sm_scale=b.sm_scale, rows=rows)


def _tree(seed, P, g, B=13, q_dtype="bf16"):
    rng = np.random.default_rng(seed)
    # level 0: one root; level 1: three branches; level 2: a node per request (some empty)
    c1 = [5, 0, 8] if B == 13 else [B // 3, B - 2 * (B // 3), B // 3]
    lengths = rng.integers(0, 150, size=B).tolist()
    return wl.make_tree(seed=seed, levels=[([B], [300]), (c1, [129, 7, 64]),
                                           ([1] * B, rng.integers(0, 40, size=B).tolist())],
                        lengths=lengths, num_qo_heads=2 * g, num_kv_heads=2, page_size=P, q_dtype=q_dtype,
                        kv_dtype=q_dtype, device="cuda")


@pytest.mark.parametrize("P", [1, 16, 64, 128])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_tree_matches_oracle(P, g):
    b = _tree(1100 + P + g, P, g)
    out, lse = _gpu_tree(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_tree_growing_scores():
    """A root whose keys grow in norm page by page, so the shared level's
    running maximum rises by more than the lazy-rescale threshold many times
    within one key-range piece (O rescaled in TMEM), next to branches and
    own pages of ordinary scale."""
    b = _tree(1160, 16, 4)
    ri, ki, idx, last = b.levels[0]
    for pos, pid in enumerate(np.asarray(idx)[ki[0]:ki[1]].tolist()):
        b.k_cache[pid] *= 1.0 + 0.5 * pos
    # one key-range piece per level (three levels), so the root's three key
    # tiles run in one CTA
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=3)
    out, lse = _gpu_tree(b, plan=plan)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_tree_f16_and_one_level():
    b = _tree(1150, 16, 4, q_dtype="f16")
    out, lse = _gpu_tree(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)
    b.levels = b.levels[:1]  # a single shared level: plain cascade
    out, lse = _gpu_tree(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("root", ["two nodes", "no keys", "no own pages"])
def test_tree_root_variants(root):
    """Root levels of other shapes: a first level of two nodes, a batch-wide
    root without keys (a level of empty states), and a batch-wide root over
    requests without own pages (no decode grid: the tree kernel and the merge
    alone)."""
    B = 13
    rng = np.random.default_rng(1170)
    lengths = rng.integers(0, 150, size=B).tolist()
    lv0 = ([6, 7], [300, 200]) if root == "two nodes" else ([B], [0 if root == "no keys" else 300])
    if root == "no own pages":
        lengths = [0] * B
    b = wl.make_tree(seed=1170, levels=[lv0, ([5, 0, 8], [129, 7, 64])], lengths=lengths, num_qo_heads=8,
                     num_kv_heads=2, page_size=16, device="cuda")
    out, lse = _gpu_tree(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref, what=root)
    assert_lse_close(lse, l_ref, what=root)


def test_tree_with_empty_level_and_many_query_tiles():
    """300 requests x g = 8 rows: a node spans several 128-row tiles, and a
    level whose nodes have no keys merges as the identity."""
    B = 300
    b = wl.make_tree(seed=1160, levels=[([B], [517]), ([100, 200], [0, 0]), ([150, 150], [33, 1])],
                     lengths=np.random.default_rng(3).integers(0, 20, size=B).tolist(), num_qo_heads=16,
                     num_kv_heads=2, page_size=16, device="cuda")
    out, lse = _gpu_tree(b)
    rows = sample_rows(b, 96, seed=4)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_tree_hnd_equals_nhd():
    from tests.test_gpu_hnd import to_hnd

    b = _tree(1170, 16, 4)
    out_n, lse_n = _gpu_tree(b)
    out_h, lse_h = _gpu_tree(b, layout="HND", kc=to_hnd(b.k_cache), vc=to_hnd(b.v_cache))
    assert torch.equal(out_h, out_n) and torch.equal(lse_h, lse_n)


def test_tree_serving_size_sampled():
    """256 requests under a 4096-key root, 16 branches of 1024 keys and
    64-512-key suffixes (GQA 32/8, bf16, page 16)."""
    b = wl.make_config_tree(device="cuda")
    out, lse = _gpu_tree(b)
    rows = sample_rows(b, 48, seed=5)
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_tree_graph_replays_after_replan():
    """A graph captured around tree_decode replays the latest plans; the
    page-index buffers are the same device arrays across the re-plans (the
    captured launches keep the pointers they were captured with)."""
    b = _tree(1180, 16, 4)
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    idx = _cuda_i32(b.kv_page_indices)
    lv = _dev_levels(b)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size)
    plan.plan_tree(lv)
    plan.tree_decode(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    out = torch.empty_like(b.q)
    lse = torch.empty(b.batch, b.num_qo_heads, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.tree_decode(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, out=out, lse=lse)
    # a new q and the same tree: replay after re-planning gives the new result
    b.q.copy_(torch.randn_like(b.q.float()).to(b.q.dtype))
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size)
    plan.plan_tree(lv)
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_tree_bad_arguments():
    b = _tree(1190, 16, 4)
    plan = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=16)
    with pytest.raises(pkd.PkdError):  # before plan
        plan.plan_tree(_dev_levels(b))
    plan.plan(b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, 16)
    bad = list(_dev_levels(b))
    ri, ki, idx, last = bad[1]
    bad[1] = (np.array([0, 5, 12], np.int32), ki[:3], idx, last[:2])  # nodes stop short of the batch
    with pytest.raises(pkd.PkdError):
        plan.plan_tree(bad)
    with pytest.raises(pkd.PkdError):  # tree_decode before plan_tree
        plan.tree_decode(b.q, b.k_cache, b.v_cache)
    small = pkd.Plan(b.batch, b.num_qo_heads, b.num_kv_heads, max_prefix_splits=2)
    small.plan(b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, 16)
    with pytest.raises(pkd.PkdError):  # three levels need three pieces
        small.plan_tree(_dev_levels(b))
