"""Invariants of the split-KV plan rule (pure-Python restatement)."""
import numpy as np
import pytest

from oracle import plan_rule


def _check(plan, indptr, last, Hk, P, G):
    B = len(indptr) - 1
    ck = plan.chunk_keys
    lens = plan.kv_len
    for b in range(B):
        n = indptr[b + 1] - indptr[b]
        assert lens[b] == (0 if n == 0 else (n - 1) * P + last[b])
    chunks = [(L + ck - 1) // ck for L in lens]
    covered = {}
    for i, (r, c0, c1, cta) in enumerate(plan.items):
        assert 0 <= c0 < c1 <= chunks[r // Hk]
        assert c1 - c0 <= max(plan.quota, 1)
        assert 0 <= cta < G
        for c in range(c0, c1):
            assert (r, c) not in covered
            covered[(r, c)] = i
    assert len(covered) == Hk * sum(chunks)
    # items in list order: rows ascending, chunks ascending within a row, CTAs non-decreasing
    keys = [(int(r), int(c0)) for r, c0, _, _ in plan.items]
    assert keys == sorted(keys)
    assert list(plan.items[:, 3]) == sorted(plan.items[:, 3])
    # per-CTA load is at most the quota
    load = np.zeros(G, np.int64)
    for r, c0, c1, cta in plan.items:
        load[cta] += c1 - c0
    assert load.max(initial=0) <= plan.quota
    # CTA ranges
    assert plan.cta_item_begin[0] == 0 and plan.cta_item_begin[-1] == len(plan.items)
    for c in range(G):
        for i in range(plan.cta_item_begin[c], plan.cta_item_begin[c + 1]):
            assert plan.items[i, 3] == c
    # row ranges
    for r in range(B * Hk):
        beg, cnt = plan.row_item_begin[r], plan.row_item_count[r]
        for i in range(beg, beg + cnt):
            assert plan.items[i, 0] == r
    assert list(plan.merge_rows) == [r for r in range(B * Hk) if plan.row_item_count[r] != 1]
    assert len(plan.items) <= G + B * Hk


@pytest.mark.parametrize("P", [1, 16, 48, 64, 128])
@pytest.mark.parametrize("G", [1, 7, 304])
def test_plan_rule_invariants(P, G):
    rng = np.random.default_rng(P * 1000 + G)
    B, Hk = 9, 3
    lens = rng.integers(0, 900, size=B)
    lens[2] = 0
    lens[5] = 1
    n = (lens + P - 1) // P
    indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
    plan = plan_rule.make_plan(indptr, last, Hk, P, G)
    _check(plan, indptr, last, Hk, P, G)
    again = plan_rule.make_plan(indptr, last, Hk, P, G)
    assert np.array_equal(plan.items, again.items)


def test_plan_rule_hand_example():
    """Two requests of 64 and 200 keys, one kv head, page 16, 3 CTAs:
    chunks 1 and 4 -> W = 5, quota 2 -> CTA0 {r0 c0, r1 c0}, CTA1 {r1 c1-2}, CTA2 {r1 c3}."""
    plan = plan_rule.make_plan([0, 4, 17], [16, 8], 1, 16, 3)
    assert plan.items.tolist() == [[0, 0, 1, 0], [1, 0, 1, 0], [1, 1, 3, 1], [1, 3, 4, 2]]
    assert plan.cta_item_begin.tolist() == [0, 2, 3, 4]
    assert plan.merge_rows.tolist() == [1]


def test_plan_rule_rejects_bad_page_size():
    with pytest.raises(ValueError):
        plan_rule.make_plan([0, 1], [5], 1, 96, 4)
