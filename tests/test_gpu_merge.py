"""GPU parity of merge_state / merge_states against the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("D", [128, 64, 8, 1024, 24])
def test_merge_state(dtype, D):
    g = torch.Generator(device="cuda").manual_seed(D)
    n, H = 257, 5
    va = torch.randn(n, H, D, device="cuda", generator=g).to(dtype)
    vb = torch.randn(n, H, D, device="cuda", generator=g).to(dtype)
    sa = torch.randn(n, H, device="cuda", generator=g) * 4
    sb = torch.randn(n, H, device="cuda", generator=g) * 4
    sa[0, 0] = -float("inf")
    sb[1, 1] = -float("inf")
    sa[2, 2] = sb[2, 2] = -float("inf")
    v, s = pkd.merge_state(va, sa, vb, sb)
    v_ref, s_ref = orc.merge_state(va.cpu(), sa.cpu(), vb.cpu(), sb.cpu())
    assert_o_close(v, v_ref)
    assert_lse_close(s, s_ref)
    assert torch.all(v[2, 2] == 0) and torch.isneginf(s[2, 2])


def test_merge_state_in_place():
    g = torch.Generator(device="cuda").manual_seed(3)
    va = torch.randn(64, 4, 128, device="cuda", generator=g)
    vb = torch.randn(64, 4, 128, device="cuda", generator=g)
    sa = torch.randn(64, 4, device="cuda", generator=g)
    sb = torch.randn(64, 4, device="cuda", generator=g)
    v_ref, s_ref = orc.merge_state(va.cpu(), sa.cpu(), vb.cpu(), sb.cpu())
    pkd.merge_state(va, sa, vb, sb, out=va, s_out=sa)
    assert_o_close(va, v_ref)
    assert_lse_close(sa, s_ref)


def test_merge_state_unaligned_rows():
    """Views that start 2 elements into their storage: the kernel takes its
    scalar path (the four-wide one needs 16-byte aligned arrays)."""
    g = torch.Generator(device="cuda").manual_seed(5)
    base_a = torch.randn(40 * 3 * 128 + 2, device="cuda", generator=g).bfloat16()
    base_b = torch.randn(40 * 3 * 128 + 2, device="cuda", generator=g).bfloat16()
    va = base_a[2:].view(40, 3, 128)
    vb = base_b[2:].view(40, 3, 128)
    sa = torch.randn(40, 3, device="cuda", generator=g)
    sb = torch.randn(40, 3, device="cuda", generator=g)
    v, s = pkd.merge_state(va, sa, vb, sb)
    v_ref, s_ref = orc.merge_state(va.cpu(), sa.cpu(), vb.cpu(), sb.cpu())
    assert_o_close(v, v_ref)
    assert_lse_close(s, s_ref)


@pytest.mark.parametrize("k", [0, 1, 3, 4, 5, 9])
def test_merge_states(k):
    g = torch.Generator(device="cuda").manual_seed(k)
    n, H, D = 33, 6, 128
    v = torch.randn(n, k, H, D, device="cuda", generator=g).bfloat16()
    s = torch.randn(n, k, H, device="cuda", generator=g) * 3
    if k:
        s[0, :, 0] = -float("inf")
    vo, so = pkd.merge_states(v, s)
    if k == 0:
        assert torch.all(vo == 0) and torch.all(torch.isneginf(so))
        return
    v_ref, s_ref = orc.merge_states(v.cpu(), s.cpu())
    assert_o_close(vo, v_ref)
    assert_lse_close(so, s_ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_merge_state_more_chunks_than_resident_threads(dtype):
    """A few times more 16-byte chunks than the one-wave grid has threads, so
    every thread strides over several, with a ragged last pass."""
    g = torch.Generator(device="cuda").manual_seed(41)
    n, H, D = 1031, 32, 128
    va = torch.randn(n, H, D, device="cuda", generator=g).to(dtype)
    vb = torch.randn(n, H, D, device="cuda", generator=g).to(dtype)
    sa = torch.randn(n, H, device="cuda", generator=g) * 4
    sb = torch.randn(n, H, device="cuda", generator=g) * 4
    sa[-1, -1] = -float("inf")
    v, s = pkd.merge_state(va, sa, vb, sb)
    v_ref, s_ref = orc.merge_state(va.cpu(), sa.cpu(), vb.cpu(), sb.cpu())
    assert_o_close(v, v_ref)
    assert_lse_close(s, s_ref)


@pytest.mark.parametrize("k,dtype", [(4, torch.bfloat16), (6, torch.bfloat16), (3, torch.float32)])
def test_merge_states_more_chunks_than_resident_threads(k, dtype):
    g = torch.Generator(device="cuda").manual_seed(43 + k)
    n, H, D = 517, 32, 128
    v = torch.randn(n, k, H, D, device="cuda", generator=g).to(dtype)
    s = torch.randn(n, k, H, device="cuda", generator=g) * 3
    s[-1, :, -1] = -float("inf")
    s[5, 0, 7] = -float("inf")
    vo, so = pkd.merge_states(v, s)
    v_ref, s_ref = orc.merge_states(v.cpu(), s.cpu())
    assert_o_close(vo, v_ref)
    assert_lse_close(so, s_ref)
    assert torch.all(vo[-1, -1] == 0) and torch.isneginf(so[-1, -1])
