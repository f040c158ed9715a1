"""GPU parity of MLA decode (latent 512 + RoPE 64, every head attending one
shared latent row per key) on the tensor cores, against the oracle: lengths
around the 32-key tile and the page, requests cut into several key ranges
and merged, head counts below and at 128, page sizes, empty requests, the
64-request DeepSeek-V3 serving workload on sampled rows, and argument checks."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import mla as orc
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def _gpu(b):
    idx = torch.as_tensor(np.asarray(b.kv_page_indices, np.int32)).cuda()
    out, lse, ws = pkd.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, idx, b.kv_last_page_len,
                                  sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    err = int(ws[:4].view(torch.int32).item())
    assert err == 0, err
    return out, lse


def _oracle(b, rows=None):
    return orc.mla_decode(b.q_nope, b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, b.kv_page_indices,
                          b.kv_last_page_len, sm_scale=b.sm_scale, rows=rows)


@pytest.mark.parametrize("P", [1, 16, 32, 64, 128])
@pytest.mark.parametrize("H", [1, 8, 16, 128])
def test_mla_matches_oracle(P, H):
    lengths = [1, 31, 32, 33, 100, 0, 777, 2100]
    b = wl.make_mla(seed=1300 + P + H, lengths=lengths, num_heads=H, page_size=P, device="cuda")
    out, lse = _gpu(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_mla_few_keys_many_requests():
    """1-3 keys per request: P's precision in the P V product shows at full size."""
    lengths = np.random.default_rng(13).integers(1, 4, size=150).tolist()
    b = wl.make_mla(seed=1350, lengths=lengths, num_heads=32, page_size=16, device="cuda")
    out, lse = _gpu(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_mla_serving_workload_sampled():
    b = wl.make_config_mla(device="cuda")
    out, lse = _gpu(b)
    rng = np.random.default_rng(2)
    rows = sorted({(int(r), int(h)) for r, h in zip(rng.integers(0, b.batch, 40), rng.integers(0, 128, 40))}
                  | {(int(np.argmax(b.kv_lens)), 0), (b.batch - 1, 127)})
    o_ref, l_ref = _oracle(b, rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_mla_is_deterministic():
    b = wl.make_mla(seed=1360, lengths=[5000, 17, 3000], num_heads=128, page_size=16, device="cuda")
    o1, l1 = _gpu(b)
    o2, l2 = _gpu(b)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mla_bad_arguments():
    b = wl.make_mla(seed=1370, lengths=[10], num_heads=16, page_size=16, device="cuda")
    idx = torch.as_tensor(np.asarray(b.kv_page_indices, np.int32)).cuda()
    with pytest.raises(ValueError):  # fp32 queries
        pkd.mla_decode(b.q_nope.float(), b.q_pe, b.ckv_cache, b.kpe_cache, b.kv_indptr, idx, b.kv_last_page_len)
    bad = wl.make_mla(seed=1371, lengths=[10], num_heads=16, page_size=24, device="cuda")
    with pytest.raises(pkd.PkdError):  # page size neither a divisor nor a multiple of 32
        pkd.mla_decode(bad.q_nope, bad.q_pe, bad.ckv_cache, bad.kpe_cache, bad.kv_indptr,
                       torch.as_tensor(np.asarray(bad.kv_page_indices, np.int32)).cuda(), bad.kv_last_page_len)
