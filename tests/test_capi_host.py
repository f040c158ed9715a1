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
