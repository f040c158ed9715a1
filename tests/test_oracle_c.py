"""The C oracle against the numpy oracle and against torch's element decoders."""
import numpy as np
import pytest
import torch

from oracle import attention as orc
from oracle import c_oracle
from paged_kv_decode_28_gb300 import workloads as wl


def test_decoders_exhaustive_against_torch():
    codes16 = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    for name, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        ref = codes16.view(tdt).to(torch.float64).numpy()
        got = np.array([c_oracle.decode_bits(name, i) for i in range(1 << 16)])
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), name
    ref8 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got8 = np.array([c_oracle.decode_bits("e4m3", i) for i in range(256)])
    assert ((got8 == ref8) | (np.isnan(got8) & np.isnan(ref8))).all()


@pytest.mark.parametrize("qd,kvd,P", [("f16", "f16", 16), ("bf16", "bf16", 1), ("bf16", "e4m3", 64), ("bf16", "bf16", 48)])
def test_c_oracle_equals_numpy_oracle(qd, kvd, P):
    batch = wl.make_paged(seed=21, lengths=[0, 1, P, P + 3, 200], num_qo_heads=8, num_kv_heads=2,
                          head_dim=64, page_size=P, q_dtype=qd, kv_dtype=kvd)
    args = (batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr, batch.kv_page_indices,
            batch.kv_last_page_len)
    kw = dict(sm_scale=batch.sm_scale, k_scale=batch.k_scale, v_scale=batch.v_scale)
    o1, l1 = orc.paged_decode(*args, **kw)
    o2, l2 = c_oracle.paged_decode(*args, **kw)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-12)


def test_c_oracle_row_subset():
    batch = wl.make_paged(seed=22, lengths=[30, 70], num_qo_heads=4, num_kv_heads=4, head_dim=32,
                          page_size=16, q_dtype="bf16", kv_dtype="bf16")
    rows = [(1, 3), (0, 0)]
    o, l = c_oracle.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                                 batch.kv_page_indices, batch.kv_last_page_len, rows=rows)
    o_all, l_all = orc.paged_decode(batch.q, batch.k_cache, batch.v_cache, batch.kv_indptr,
                                    batch.kv_page_indices, batch.kv_last_page_len)
    for b, h in rows:
        np.testing.assert_allclose(o[b, h], o_all[b, h], rtol=1e-12, atol=1e-12)
    assert np.isnan(l[0, 1])
