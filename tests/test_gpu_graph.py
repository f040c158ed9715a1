"""CUDA-graph friendliness: run() captured once keeps its launch shape, and a
re-plan of new lengths followed by a replay equals an eager run."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import gpu_paged_decode

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
        eager = pkd.Plan(B, Hq, Hk)
        eager.plan(indptr, idx, last, P)
        o2, l2 = eager.run(q, pool.k_cache, pool.v_cache)
        torch.cuda.synchronize()
        assert torch.equal(out, o2), trial
        assert torch.equal(lse, l2), trial
