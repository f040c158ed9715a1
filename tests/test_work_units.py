"""Host logic of the work lists (no GPU): the units pkd_plan_prefill,
pkd_plan_tree and pkd_mla_decode upload, built by the library's host-only
exports and checked against what the kernels rely on -- both units of a pair
share their keys, every query row is covered exactly once, a node's or a
request's key-range pieces partition its keys, the causal key range is the one
the pair's last row sees, MLA's piece size is the smallest that fits the SMs,
and pairs come longest first (prefill: a request's pairs together, longest
first, requests in order of their longest pair)."""
import numpy as np
import pytest

import paged_kv_decode_28_gb300 as pkd
from paged_kv_decode_28_gb300 import _build, api

NO_CAUSAL = 2**31 - 1
Q0, QEND, PB, KVLEN, T0, T1, PIECE, LEVEL, DIAG = range(9)


@pytest.fixture(scope="module", autouse=True)
def _library():
    _build.build()  # host-only entry points: no GPU needed


def _pairs(u):
    assert len(u) % 2 == 0
    return [(u[2 * j], u[2 * j + 1]) for j in range(len(u) // 2)]


def _rows(a, per_tile):
    return range(a[Q0], min(a[Q0] + per_tile, a[QEND]))


def _check_pair_invariants(u, per_tile, by_request=False):
    for a, b in _pairs(u):
        for f in (QEND, PB, KVLEN, T0, T1, PIECE, LEVEL, DIAG):
            assert a[f] == b[f], f
        assert a[Q0] < a[QEND]  # the first tile always has rows
        assert b[Q0] == min(a[Q0] + per_tile, a[QEND])
    lengths = [a[T1] - a[T0] for a, _ in _pairs(u)]
    if not by_request:
        assert lengths == sorted(lengths, reverse=True)
        return
    # a request's pairs are contiguous and longest first; the requests come in
    # order of their longest pair
    groups = []
    for a, _ in _pairs(u):
        key = (a[PB], a[QEND])
        if not groups or groups[-1][0] != key:
            assert all(g[0] != key for g in groups), "a request's pairs are split"
            groups.append((key, []))
        groups[-1][1].append(a[T1] - a[T0])
    for _, ls in groups:
        assert ls == sorted(ls, reverse=True)
    firsts = [ls[0] for _, ls in groups]
    assert firsts == sorted(firsts, reverse=True)


def _prefill_case(rng, B, P):
    q_lens = rng.integers(0, 300, size=B)
    kv_lens = q_lens + rng.integers(0, 700, size=B)
    pages = (kv_lens + P - 1) // P
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    kvi = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = np.where(pages > 0, kv_lens - (pages - 1) * P, 0).astype(np.int32)
    return qo, kvi, last, kv_lens


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("P", [1, 16, 64])
def test_prefill_units(causal, g, P):
    rng = np.random.default_rng(100 * g + P + causal)
    B = 9
    qo, kvi, last, kv_lens = _prefill_case(rng, B, P)
    per_tile = 128 // g
    u = api.prefill_units(qo, kvi, last, 8 * g, 8, P, causal=causal)
    _check_pair_invariants(u, per_tile, by_request=True)
    seen = np.zeros(int(qo[-1]), np.int32)
    for a, b in _pairs(u):
        r = int(np.searchsorted(qo, a[Q0], side="right")) - 1
        assert qo[r] <= a[Q0] < qo[r + 1] and a[QEND] == qo[r + 1]
        assert a[PB] == kvi[r] and a[KVLEN] == kv_lens[r]
        assert a[T0] == 0 and a[PIECE] == -1 and a[LEVEL] == 0
        for t in (a, b):
            for row in _rows(t, per_tile):
                seen[row] += 1
        if causal:
            diag = int(kv_lens[r] - (qo[r + 1] - qo[r]) - qo[r])
            assert a[DIAG] == diag
            last_tok = min(a[Q0] + 2 * per_tile, a[QEND]) - 1
            keys = last_tok + diag + 1  # keys the pair's last row sees
            assert a[T1] == (keys + 127) // 128
            assert 0 < keys <= kv_lens[r]
        else:
            assert a[DIAG] == NO_CAUSAL and a[T1] == (kv_lens[r] + 127) // 128
    assert np.all(seen == 1)  # every query token in exactly one tile


def test_prefill_units_edge_cases():
    # no query tokens: no units; a request whose query fills exactly two tiles: one full pair
    u = api.prefill_units([0, 0, 64], [0, 4, 8], [16, 16], 32, 8, 16)
    assert len(u) == 2 and u[0][Q0] == 0 and u[1][Q0] == 32 and u[0][QEND] == 64
    # one query tile: paired with an empty one
    u = api.prefill_units([0, 5], [0, 1], [9], 32, 8, 16)
    assert len(u) == 2 and u[1][Q0] == u[1][QEND] == 5 and u[0][T1] == 1
    with pytest.raises(pkd.PkdError):  # more query tokens than keys
        api.prefill_units([0, 20], [0, 1], [9], 32, 8, 16)
    with pytest.raises(pkd.PkdError):  # last_page_len outside 1..P
        api.prefill_units([0, 5], [0, 1], [17], 32, 8, 16)
    with pytest.raises(pkd.PkdError):  # a group size that does not divide 128
        api.prefill_units([0, 5], [0, 1], [9], 24, 8, 16)


def _tree_case(rng, B, P, n_levels):
    levels = []
    for l in range(n_levels):
        n_nodes = 1 if l == 0 else int(rng.integers(2, 6))
        cuts = np.sort(rng.choice(np.arange(1, B), size=n_nodes - 1, replace=False)) if n_nodes > 1 else []
        ri = np.concatenate([[0], cuts, [B]]).astype(np.int32)
        lens = rng.integers(0, 3000, size=n_nodes)
        lens[rng.integers(0, n_nodes)] = 0 if l > 0 else lens[0]  # an empty node below the root
        pages = (lens + P - 1) // P
        ki = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        last = np.where(pages > 0, lens - (pages - 1) * P, 0).astype(np.int32)
        levels.append((ri, ki, last, lens))
    return levels


@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("n_levels", [1, 2, 4])
def test_tree_units(g, n_levels):
    rng = np.random.default_rng(7 * g + n_levels)
    B, P, max_splits, num_ctas = 300, 16, 16, 304
    per_tile = 128 // g
    levels = _tree_case(rng, B, P, n_levels)
    u, pieces = api.tree_units([(ri, ki, last) for ri, ki, last, _ in levels], B, 8 * g, 8, P, num_ctas, max_splits)
    _check_pair_invariants(u, per_tile)
    assert n_levels <= pieces <= max_splits
    piece_base = 0
    for l, (ri, ki, last, lens) in enumerate(levels):
        lu = [p for p in _pairs(u) if p[0][LEVEL] == l]
        level_pieces = sorted({int(a[PIECE]) for a, _ in lu})
        S = len(level_pieces)
        assert level_pieces == list(range(piece_base, piece_base + S))  # contiguous piece ids per level
        for n in range(len(ri) - 1):
            nu = [p for p in lu if p[0][PB] == ki[n] and p[0][QEND] == ri[n + 1]
                  and ri[n] <= p[0][Q0] < ri[n + 1]]
            tiles = (int(lens[n]) + 127) // 128
            if ri[n + 1] == ri[n]:
                assert not nu  # a node without requests has no units
                continue
            for piece in level_pieces:  # every piece of every request is written
                pu = [p for p in nu if p[0][PIECE] == piece]
                seen = np.zeros(B, np.int32)
                for a, b in pu:
                    assert a[KVLEN] == lens[n] and a[DIAG] == NO_CAUSAL
                    for t in (a, b):
                        for row in _rows(t, per_tile):
                            seen[row] += 1
                assert np.all(seen[ri[n]:ri[n + 1]] == 1) and seen.sum() == ri[n + 1] - ri[n]
            # the pieces' key ranges partition the node's key tiles, in piece order
            ranges = sorted({(int(a[PIECE]), int(a[T0]), int(a[T1])) for a, _ in nu})
            assert len(ranges) == S
            assert ranges[0][1] == 0 and ranges[-1][2] == tiles
            for (_, _, e), (_, s2, _) in zip(ranges, ranges[1:]):
                assert e == s2
        piece_base += S
    assert piece_base == pieces


def test_tree_units_errors():
    lv = [([0, 4], [0, 2], [16])]
    with pytest.raises(pkd.PkdError):  # more levels than pieces
        api.tree_units(lv * 3, 4, 32, 8, 16, 304, 2)
    with pytest.raises(pkd.PkdError):  # nodes must cover the batch
        api.tree_units([([0, 3], [0, 2], [16])], 4, 32, 8, 16, 304, 4)
    with pytest.raises(pkd.PkdError):  # five levels
        api.tree_units(lv * 5, 4, 32, 8, 16, 304, 16)
    with pytest.raises(pkd.PkdError):  # last_page_len outside 1..P
        api.tree_units([([0, 4], [0, 2], [17])], 4, 32, 8, 16, 304, 4)


def _mla_piece_size(tiles, num_sms):
    """The rule the split follows, restated: the smallest C >= 16 (32-key
    tiles) whose pieces -- ceil(tiles / C) per request, at least one -- number
    at most num_sms, or the longest request's tile count when none does."""
    def pieces(C):
        return sum(max(1, -(-t // C)) for t in tiles)
    top = max(max(tiles), 1)
    C = next((c for c in range(1, top + 1) if pieces(c) <= num_sms), top)
    return max(C, 16)


@pytest.mark.parametrize("seed,B,P,num_sms", [(1, 64, 16, 152), (2, 7, 1, 148), (3, 200, 64, 152),
                                              (4, 1, 32, 152), (5, 30, 16, 8)])
def test_mla_units(seed, B, P, num_sms):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 9000, size=B)
    lens[rng.integers(0, B)] = 0  # an empty request
    pages = (lens + P - 1) // P
    kvi = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = np.where(pages > 0, lens - (pages - 1) * P, 0).astype(np.int32)
    u, rpb = pkd.mla_units(kvi, last, P, num_sms)
    tiles = [(int(L) + 31) // 32 for L in lens]
    C = _mla_piece_size(tiles, num_sms)
    halves = _pairs(u)
    for a, b in halves:  # the two output halves of one key range, side by side
        assert a[LEVEL] == 0 and b[LEVEL] == 1
        for f in (Q0, QEND, PB, KVLEN, T0, T1, PIECE):
            assert a[f] == b[f], f
    lengths = [a[T1] - a[T0] for a, _ in halves]
    assert lengths == sorted(lengths, reverse=True)
    assert rpb[0] == 0
    for r in range(B):
        ru = sorted((int(a[T0]), int(a[T1]), int(a[PIECE])) for a, _ in halves if a[Q0] == r)
        np_r = len(ru)
        assert np_r == max(1, -(-tiles[r] // C))
        assert all(a[KVLEN] == lens[r] and a[PB] == kvi[r] and a[QEND] == r + 1 for a, _ in halves if a[Q0] == r)
        # the ranges partition the request's tiles, each at most C long
        assert ru[0][0] == 0 and ru[-1][1] == tiles[r]
        for (_, e, _), (s2, _, _) in zip(ru, ru[1:]):
            assert e == s2
        assert all(t1 - t0 <= C for t0, t1, _ in ru)
        if np_r == 1:
            assert ru[0][2] == -1 and rpb[r + 1] == rpb[r]  # written directly
        else:
            assert [p for _, _, p in ru] == list(range(rpb[r], rpb[r + 1]))
    assert len(halves) <= max(num_sms, B)


def test_mla_units_errors():
    with pytest.raises(pkd.PkdError):  # last_page_len outside 1..P
        pkd.mla_units([0, 2], [17], 16, 152)
    with pytest.raises(pkd.PkdError):  # decreasing kv_indptr
        pkd.mla_units([0, 2, 1], [16, 16], 16, 152)
    with pytest.raises(pkd.PkdError):  # no SMs
        pkd.mla_units([0, 2], [16], 16, 0)


def test_units_call_retries_with_the_reported_size():
    """A too-small buffer gets PKD_ERR_CAPACITY_EXCEEDED with the needed count,
    and the binding retries once with that size."""
    import ctypes

    qo, kvi, last = [0, 500], [0, 40], [16]
    want = api.prefill_units(qo, kvi, last, 32, 8, 16)
    qi, ki, la = (np.asarray(x, np.int32) for x in (qo, kvi, last))
    calls = []

    def fn(buf, cap, n):
        calls.append(cap)
        return api.lib().pkd_prefill_units_host(api._as_i32p(qi), api._as_i32p(ki), api._as_i32p(la), 1, 32, 8, 16,
                                                1, api._as_i32p(buf), cap, ctypes.byref(n))

    got = api._units_call(fn, 1)
    assert calls == [1, len(want)] and np.array_equal(got, want)
