"""Host-side checks of the C ABI (no GPU): the library loads and exports every
symbol the header declares, and the C++ planner equals the pure-Python
restatement of the split-KV rule bit for bit."""
import os
import re

import numpy as np
import pytest

from oracle import plan_rule
import paged_kv_decode_28_gb300 as pkd
from paged_kv_decode_28_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "pkd.h")).read()
    names = sorted(set(re.findall(r"\b(pkd_[a-z_]+)\s*\(", header)))
    assert len(names) >= 14
    L = pkd.lib()
    for n in names:
        assert hasattr(L, n), n
    assert pkd.version().startswith("pkd ")


def test_binding_signatures_match_the_header():
    """Every entry point the binding declares has the header's argument count
    and 64-bit integers where the header has int64_t / size_t (a mismatch
    would pass wrong values through ctypes without any error)."""
    import ctypes

    header = open(os.path.join(ROOT, "include", "pkd.h")).read()
    protos = {}
    for m in re.finditer(r"\b(?:pkd_status|size_t|const char\*)\s+(pkd_[a-z_]+)\s*\(([^;]*?)\);", header, re.S):
        args = [a.strip() for a in m.group(2).split(",")] if m.group(2).strip() not in ("", "void") else []
        protos[m.group(1)] = args
    L = pkd.lib()
    checked = 0
    for name, args in protos.items():
        fn = getattr(L, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == len(args), (name, len(fn.argtypes), len(args))
        for decl, ct in zip(args, fn.argtypes):
            if re.match(r"(int64_t|size_t)\s+\w+$", decl):
                assert ct in (ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64), (name, decl, ct)
            elif re.match(r"int\s+\w+$", decl):
                assert ct is ctypes.c_int, (name, decl, ct)
            elif re.match(r"float\s+\w+$", decl):
                assert ct is ctypes.c_float, (name, decl, ct)
        checked += 1
    assert checked >= 20


def _random_table(rng, B, P, max_len, empty_frac=0.1):
    lens = rng.integers(1, max_len + 1, size=B)
    lens[rng.random(B) < empty_frac] = 0
    n = (lens + P - 1) // P
    indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
    return indptr, last


@pytest.mark.parametrize("seed", range(12))
def test_cpp_planner_equals_python_rule(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 3, 16, 48, 64, 128, 256]))
    B = int(rng.integers(1, 60))
    Hk = int(rng.choice([1, 2, 8]))
    G = int(rng.choice([1, 5, 152, 304]))
    indptr, last = _random_table(rng, B, P, int(rng.choice([10, 700, 5000])))
    ref = plan_rule.make_plan(indptr, last, Hk, P, G)
    got = pkd.plan_host(indptr, last, Hk, P, G)
    assert np.array_equal(got["items"], ref.items)
    assert np.array_equal(got["cta_item_begin"], ref.cta_item_begin)
    assert np.array_equal(got["row_item_begin"], ref.row_item_begin)
    assert np.array_equal(got["row_item_count"], ref.row_item_count)
    assert np.array_equal(got["merge_rows"], ref.merge_rows)
    assert got["chunk_keys"] == ref.chunk_keys and got["quota"] == ref.quota


def test_planner_on_standard_workload_tables():
    from paged_kv_decode_28_gb300 import workloads as wl
    for idx in (1, 2, 3, 4, 5):
        lens = wl.config_lengths(idx)
        P = 64 if idx == 5 else 16
        n = (lens + P - 1) // P
        indptr = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        last = np.where(n > 0, lens - (n - 1) * P, 0).astype(np.int32)
        Hk = 32 if idx == 1 else 8
        ref = plan_rule.make_plan(indptr, last, Hk, P, 304)
        got = pkd.plan_host(indptr, last, Hk, P, 304)
        assert np.array_equal(got["items"], ref.items)
        assert np.array_equal(got["cta_item_begin"], ref.cta_item_begin)
        # balance: no CTA holds more than the quota
        load = np.zeros(304, np.int64)
        for r, c0, c1, cta in got["items"]:
            load[cta] += c1 - c0
        assert load.max() == ref.quota


@pytest.mark.parametrize("indptr,last,P,status", [
    ([1, 3], [4], 16, 1),          # indptr[0] != 0
    ([0, 3, 2], [4, 4], 16, 1),    # decreasing
    ([0, 3], [0], 16, 1),          # last page empty
    ([0, 3], [17], 16, 1),         # last page longer than a page
    ([0, 1], [5], 96, 2),          # page size above 64 but not a multiple of 64
    ([0, 1], [5], 0, 2),           # page size 0
])
def test_planner_rejects_bad_tables(indptr, last, P, status):
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host(indptr, last, 2, P, 8)
    assert e.value.status == status


def test_workspace_bytes_rules():
    L = pkd.lib()
    assert L.pkd_workspace_bytes(64, 32, 8, 128, 304, 0) > 0
    assert L.pkd_workspace_bytes(64, 32, 8, 64, 304, 0) == 0       # head_dim 64 not built
    assert L.pkd_workspace_bytes(64, 30, 8, 128, 304, 0) == 0       # not a multiple
    assert L.pkd_workspace_bytes(64, 32, 8, 128, 304, 17) == 0      # too many prefix splits
    assert L.pkd_workspace_bytes(64, 32, 8, 128, 304, 4) > L.pkd_workspace_bytes(64, 32, 8, 128, 304, 0)


def test_plan_create_validates_without_a_gpu():
    import ctypes
    L = pkd.lib()
    h = ctypes.c_void_p()
    # group of 16 is above the built maximum of 8
    st = L.pkd_plan_create(ctypes.byref(h), 4, 64, 4, 128, 8, 0, ctypes.c_void_p(256), 1 << 30)
    assert st == 2
    # a workspace that is too small
    st = L.pkd_plan_create(ctypes.byref(h), 4, 32, 8, 128, 8, 0, ctypes.c_void_p(256), 16)
    assert st == 3
    # misaligned workspace
    st = L.pkd_plan_create(ctypes.byref(h), 4, 32, 8, 128, 8, 0, ctypes.c_void_p(260), 1 << 30)
    assert st == 1
    st = L.pkd_plan_create(ctypes.byref(h), 4, 32, 8, 128, 8, 0, ctypes.c_void_p(256), 1 << 30)
    assert st == 0
    assert L.pkd_plan_destroy(h) == 0


def test_next_row_entry_points_validate_without_a_gpu():
    """Argument checks of the append, layout, tree, prefill and MLA entry points
    run on the host before any CUDA call (status codes as in pkd.h)."""
    import ctypes
    L = pkd.lib()
    OK, INVALID, UNSUPPORTED, SMALL, NO_PLAN = 0, 1, 2, 3, 7
    p16 = ctypes.c_void_p(1 << 20)  # a 16-byte aligned stand-in address, never dereferenced
    one = np.array([0, 1], np.int32)
    last = np.array([1], np.int32)
    i32 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    # KV append: no tokens is a no-op; head_dim, dtype pairing, scales, layout and alignment are checked
    args = lambda **kw: dict(dict(k=p16, v=p16, nd=1, bi=p16, pos=p16, n=4, ip=p16, idx=p16, B=1, Hk=2, D=128, P=16,
                                  kc=p16, vc=p16, kd=1, lay=0, N=8, stride=16 * 2 * 128, ks=None, vs=None), **kw)
    call = lambda a: L.pkd_append_kv(a["k"], a["v"], a["nd"], a["bi"], a["pos"], a["n"], a["ip"], a["idx"], a["B"],
                                     a["Hk"], a["D"], a["P"], a["kc"], a["vc"], a["kd"], a["lay"], a["N"], a["stride"],
                                     a["ks"], a["vs"], None, None)
    assert call(args(n=0)) == OK
    assert call(args(D=64)) == UNSUPPORTED
    assert call(args(nd=0)) == UNSUPPORTED                 # f16 values into a bf16 pool
    assert call(args(kd=2, stride=16 * 2 * 128)) == INVALID  # an e4m3 pool needs scales
    assert call(args(lay=2)) == INVALID
    assert call(args(kc=ctypes.c_void_p((1 << 20) + 8))) == INVALID
    assert call(args(stride=100)) == INVALID

    # the page layout of a plan
    h = ctypes.c_void_p()
    assert L.pkd_plan_create(ctypes.byref(h), 4, 32, 8, 128, 8, 2, ctypes.c_void_p(256), 1 << 30) == OK
    assert L.pkd_plan_set_kv_layout(h, 2) == INVALID
    assert L.pkd_plan_set_kv_layout(h, 1) == OK
    # prefix tree and its decode before a plan of the requests' own pages
    lv = (ctypes.c_void_p * 1)(one.ctypes.data)
    pg = (ctypes.c_void_p * 1)(p16.value)
    nn = np.array([1], np.int32)
    assert L.pkd_plan_tree(h, 1, lv, lv, pg, (ctypes.c_void_p * 1)(last.ctypes.data), i32(nn), None) == NO_PLAN
    assert L.pkd_tree_decode(h, p16, p16, p16, 8, 16 * 8 * 128, 0.0, p16, None, None) == NO_PLAN
    # prefill: head counts must be the plan's, K/V 16-bit of q's type, q_len <= kv_len
    qo = np.array([0, 5], np.int32)
    assert L.pkd_plan_prefill(h, i32(qo), i32(one), p16, i32(last), 1, 16, 8, 128, 16, 1, 1, 1, None) == INVALID
    assert L.pkd_plan_prefill(h, i32(qo), i32(one), p16, i32(last), 1, 32, 8, 128, 16, 1, 2, 1, None) == UNSUPPORTED
    assert L.pkd_plan_prefill(h, i32(qo), i32(one), p16, i32(last), 1, 32, 8, 128, 16, 1, 1, 1, None) == INVALID
    assert L.pkd_prefill_run(h, p16, p16, p16, 8, 16 * 8 * 128, 0.0, p16, None, None) == NO_PLAN
    assert L.pkd_plan_destroy(h) == OK

    # MLA: workspace rule and argument checks
    assert L.pkd_mla_workspace_bytes(64, 128, 148) > L.pkd_mla_workspace_bytes(64, 16, 148) > 0
    assert L.pkd_mla_workspace_bytes(64, 129, 148) == 0
    assert L.pkd_mla_workspace_bytes(64, 128, 0) == 0
    need = L.pkd_mla_workspace_bytes(1, 16, 148)
    mla = lambda P=16, H=16, ws=need, B=1: L.pkd_mla_decode(p16, p16, p16, p16, i32(one), p16, i32(last), B, H, P, 8,
                                                           P * 512, P * 64, 0.0, p16, None, p16, ws, 148, None)
    assert mla(P=24) == UNSUPPORTED
    assert mla(H=200) == UNSUPPORTED
    assert mla(ws=need - 256) == SMALL
    assert mla(B=0) == OK
