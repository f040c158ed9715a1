"""GPU parity of pkd_append_kv (new tokens' K/V written into the paged cache)
against the CPU oracle: bit-exact pools for 16-bit copies and for e4m3 codes,
skipped out-of-table tokens with the device flag, and decode after append
equal to the oracle over the longer sequences."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from oracle import kv_append as ka
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close, gpu_paged_decode

pytestmark = pytest.mark.gpu


def _cuda_i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _batch(seed, lens, P, kvd, Hq=16, Hk=4):
    # tables sized for one more token per request: the appended one
    return wl.make_paged(seed=seed, lengths=(np.asarray(lens) + 1).tolist(), num_qo_heads=Hq, num_kv_heads=Hk,
                         page_size=P, kv_dtype=kvd, q_dtype="bf16", device="cuda")


@pytest.mark.parametrize("kvd,newd", [("bf16", torch.bfloat16), ("f16", torch.float16), ("e4m3", torch.bfloat16),
                                      ("e4m3", torch.float16)])
@pytest.mark.parametrize("P", [1, 16, 64])
def test_append_matches_oracle_bit_for_bit(kvd, newd, P):
    lens = np.array([0, 5, 15, 16, 63, 64, 200])
    b = _batch(800 + P, lens, P, kvd)
    if kvd == "f16":
        b.q = b.q.to(torch.float16)
    gen = torch.Generator(device="cuda").manual_seed(5)
    n, Hk = len(lens), b.num_kv_heads
    # scaled so that some e4m3 quotients exceed 448 (saturation) and some are tiny (subnormals)
    k_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(newd)
    v_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(newd)
    if kvd == "e4m3":
        k_new[0, 0, :4] = torch.tensor([6e4, -6e4, 1e-6, 0.0], dtype=newd)
    kr, vr, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, np.arange(n), lens, b.kv_indptr,
                                   b.kv_page_indices, P, b.k_scale, b.v_scale)
    assert skipped == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(k_new, v_new, _cuda_i32(np.arange(n)), _cuda_i32(lens), _cuda_i32(b.kv_indptr),
                  _cuda_i32(b.kv_page_indices), b.k_cache, b.v_cache, k_scale=b.k_scale, v_scale=b.v_scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    view = (lambda t: t.view(torch.uint8)) if kvd == "e4m3" else (lambda t: t)
    assert torch.equal(view(b.k_cache.cpu()), view(kr)) and torch.equal(view(b.v_cache.cpu()), view(vr))


@pytest.mark.parametrize("newd", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("scale", [1.7, 3.0, 0.37, 0.0123, 1e-3])
def test_e4m3_codes_of_every_16_bit_value(newd, scale):
    """Every finite bf16 / f16 value through the e4m3 path: the codes must be
    those of the fp32 quotient x / scale.  Scales such as 3 put quotients
    exactly on rounding midpoints (x = 3 * midpoint), where the quotient's
    tie-to-even decides and a reciprocal multiply alone lands on the wrong side
    for some of them (1.7); tiny scales overflow the quotient."""
    allv = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(newd)
    vals = allv[torch.isfinite(allv)]
    Hk, P = 2, 16
    per = Hk * 128
    n = (vals.numel() + per - 1) // per
    flat = torch.zeros(n * per, dtype=newd)
    flat[:vals.numel()] = vals
    k_new = flat.view(n, Hk, 128).cuda()
    v_new = (-flat).view(n, Hk, 128).cuda()  # the negative half again, in the other table
    pages = (n + P - 1) // P
    b = wl.make_paged(seed=840, lengths=[n], num_qo_heads=4, num_kv_heads=Hk, page_size=P, kv_dtype="e4m3",
                      pool_pages=pages, device="cuda")
    k_scale = torch.tensor([scale, scale * 1.25], dtype=torch.float32, device="cuda")
    v_scale = torch.tensor([scale * 0.75, scale], dtype=torch.float32, device="cuda")
    pos = np.arange(n)
    kr, vr, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, np.zeros(n, np.int64), pos, b.kv_indptr,
                                   b.kv_page_indices, P, k_scale, v_scale)
    assert skipped == 0
    pkd.append_kv(k_new, v_new, _cuda_i32(np.zeros(n, np.int64)), _cuda_i32(pos), _cuda_i32(b.kv_indptr),
                  _cuda_i32(b.kv_page_indices), b.k_cache, b.v_cache, k_scale=k_scale, v_scale=v_scale)
    torch.cuda.synchronize()
    assert torch.equal(b.k_cache.cpu().view(torch.uint8), kr.view(torch.uint8))
    assert torch.equal(b.v_cache.cpu().view(torch.uint8), vr.view(torch.uint8))


@pytest.mark.parametrize("kvd", ["bf16", "e4m3"])
def test_append_more_tokens_than_resident_warps(kvd):
    """More new tokens than the one-wave grid has warps (each warp strides over
    several tokens), appended at the end of a few long requests."""
    P, Hk = 16, 2
    reqs, per = 4, 2503
    lens = np.full(reqs, per, dtype=np.int64)
    b = wl.make_paged(seed=870, lengths=lens.tolist(), num_qo_heads=4, num_kv_heads=Hk, page_size=P, kv_dtype=kvd,
                      q_dtype="bf16", device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(9)
    n = reqs * per
    k_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(torch.bfloat16)
    v_new = (torch.randn(n, Hk, 128, device="cuda", generator=gen) * 3).to(torch.bfloat16)
    bi = np.repeat(np.arange(reqs), per)
    pos = np.tile(np.arange(per), reqs)  # every slot of every request, rewritten
    kr, vr, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, bi, pos, b.kv_indptr, b.kv_page_indices, P,
                                   b.k_scale, b.v_scale)
    assert skipped == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(k_new, v_new, _cuda_i32(bi), _cuda_i32(pos), _cuda_i32(b.kv_indptr), _cuda_i32(b.kv_page_indices),
                  b.k_cache, b.v_cache, k_scale=b.k_scale, v_scale=b.v_scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    view = (lambda t: t.view(torch.uint8)) if kvd == "e4m3" else (lambda t: t)
    assert torch.equal(view(b.k_cache.cpu()), view(kr)) and torch.equal(view(b.v_cache.cpu()), view(vr))


def test_append_then_decode_equals_oracle():
    lens = np.array([1, 17, 300, 64, 1000])
    for kvd in ("bf16", "e4m3"):
        b = _batch(820, lens, 16, kvd, Hq=32, Hk=8)
        gen = torch.Generator(device="cuda").manual_seed(6)
        n, Hk = len(lens), b.num_kv_heads
        k_new = torch.randn(n, Hk, 128, device="cuda", generator=gen).to(torch.bfloat16)
        v_new = torch.randn(n, Hk, 128, device="cuda", generator=gen).to(torch.bfloat16)
        pkd.append_kv(k_new, v_new, _cuda_i32(np.arange(n)), _cuda_i32(lens), _cuda_i32(b.kv_indptr),
                      _cuda_i32(b.kv_page_indices), b.k_cache, b.v_cache, k_scale=b.k_scale, v_scale=b.v_scale)
        out, lse, _ = gpu_paged_decode(b)
        o_ref, l_ref = orc.paged_decode(b.q, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                                        b.kv_last_page_len, sm_scale=b.sm_scale, k_scale=b.k_scale,
                                        v_scale=b.v_scale)
        assert_o_close(out, o_ref)
        assert_lse_close(lse, l_ref)


def test_out_of_table_tokens_are_skipped_and_flagged():
    P = 16
    lens = np.array([16, 5])
    b = wl.make_paged(seed=830, lengths=lens.tolist(), num_qo_heads=4, num_kv_heads=2, page_size=P,
                      pool_pages=8, device="cuda")
    before_k, before_v = b.k_cache.clone(), b.v_cache.clone()
    k_new = torch.ones(4, 2, 128, dtype=torch.bfloat16, device="cuda")
    bi, pos = [0, 1, 2, 0], [16, 3, 0, -1]
    kr, vr, skipped = ka.append_kv(before_k, before_v, k_new, k_new, bi, pos, b.kv_indptr, b.kv_page_indices, P)
    assert skipped == 3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(k_new, k_new, _cuda_i32(bi), _cuda_i32(pos), _cuda_i32(b.kv_indptr), _cuda_i32(b.kv_page_indices),
                  b.k_cache, b.v_cache, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkd.api.DEVERR_PAGE_INDEX
    assert torch.equal(b.k_cache.cpu(), kr) and torch.equal(b.v_cache.cpu(), vr)


def test_append_rejects_bad_arguments():
    b = wl.make_paged(seed=840, lengths=[3], num_qo_heads=2, num_kv_heads=1, page_size=16, device="cuda")
    k_new = torch.zeros(1, 1, 128, dtype=torch.float16, device="cuda")  # f16 into a bf16 pool
    with pytest.raises(pkd.PkdError):
        pkd.append_kv(k_new, k_new, _cuda_i32([0]), _cuda_i32([3]), _cuda_i32(b.kv_indptr),
                      _cuda_i32(b.kv_page_indices), b.k_cache, b.v_cache)
