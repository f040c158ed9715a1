"""Pins of the KV-append oracle (oracle/kv_append.py) against facts it does not
compute itself: E4M3 codes worked out from the format's bit layout (1 sign, 4
exponent bits with bias 7, 3 mantissa bits, subnormals, 0x7F / 0xFF NaN),
round-to-nearest-even ties, saturation, a round trip over every finite code,
and decode attention after an append equal to library attention over the
concatenated keys."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as orc
from oracle import kv_append as ka
from paged_kv_decode_28_gb300 import workloads as wl


def _e4m3_value(code: int) -> float:
    """E4M3 value from its bits (written out here, independent of torch)."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return math.nan
    if e == 0:
        return s * m * 2.0 ** -9  # subnormal: m/8 * 2^(1-7)
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_encoder_known_codes():
    cases = {1.0: 0x38, -1.0: 0xB8, 448.0: 0x7E, -448.0: 0xFE, 2.0 ** -9: 0x01, 2.0 ** -6: 0x08,
             0.0: 0x00, 1.25: 0x3A, 240.0: 0x77}
    got = ka.e4m3_encode(list(cases)).tolist()
    assert got == list(cases.values())


def test_encoder_ties_go_to_even_codes():
    # midpoints between neighbouring finite codes (same sign, positive): the
    # result is the neighbour whose mantissa (code) is even
    for c in range(0x00, 0x7E):
        lo, hi = _e4m3_value(c), _e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exactly representable in float32
        want = c if c % 2 == 0 else c + 1
        assert ka.e4m3_encode([mid])[0] == want, (c, lo, hi)


def test_encoder_saturates_and_keeps_nan():
    got = ka.e4m3_encode([449.0, 479.9, 480.0, 1e6, np.inf, -1e6, -np.inf, np.nan]).tolist()
    assert got[:5] == [0x7E] * 5 and got[5:7] == [0xFE] * 2
    assert got[7] in (0x7F, 0xFF)


def test_encoder_round_trips_every_finite_code():
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = np.array([_e4m3_value(c) for c in codes], dtype=np.float32)
    assert ka.e4m3_encode(vals).tolist() == codes


def test_decode_after_append_is_attention_over_the_longer_sequence():
    """Append one token per request at position L_b (pages allocated ahead),
    then decode over L_b + 1 keys: equals torch SDPA over old keys ++ new key."""
    P, Hq, Hk, D = 16, 8, 2, 128
    lens = np.array([15, 16, 1, 40])
    b = wl.make_paged(seed=700, lengths=(lens + 1).tolist(), num_qo_heads=Hq, num_kv_heads=Hk, page_size=P,
                      head_dim=D, pool_pages=32)
    gen = torch.Generator().manual_seed(7)
    k_new = torch.randn(len(lens), Hk, D, generator=gen).to(torch.bfloat16)
    v_new = torch.randn(len(lens), Hk, D, generator=gen).to(torch.bfloat16)
    k2, v2, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, np.arange(len(lens)), lens, b.kv_indptr,
                                   b.kv_page_indices, P)
    assert skipped == 0
    o, lse = orc.paged_decode(b.q, k2, v2, b.kv_indptr, b.kv_page_indices, b.kv_last_page_len,
                              sm_scale=b.sm_scale)
    for r in range(len(lens)):
        toks = orc.request_tokens(b.kv_indptr, b.kv_page_indices, b.kv_last_page_len, P, r)[: lens[r]]
        kk = torch.cat([torch.stack([b.k_cache[p, t] for p, t in toks]).double(), k_new[r : r + 1].double()])
        vv = torch.cat([torch.stack([b.v_cache[p, t] for p, t in toks]).double(), v_new[r : r + 1].double()])
        g = Hq // Hk
        qh = b.q[r].double().view(Hk, g, D)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qh.unsqueeze(2), kk.permute(1, 0, 2).unsqueeze(1), vv.permute(1, 0, 2).unsqueeze(1),
            scale=b.sm_scale).view(Hq, D)
        assert np.allclose(o[r], ref.numpy(), rtol=0, atol=1e-12)


def test_out_of_table_tokens_are_skipped():
    P = 16
    b = wl.make_paged(seed=701, lengths=[16, 5], num_qo_heads=2, num_kv_heads=1, page_size=P, head_dim=128,
                      pool_pages=4)
    k_new = torch.ones(4, 1, 128, dtype=torch.bfloat16)
    # request 0 has one page (positions 0..15), request 1 one page; request 2 does not exist
    k2, v2, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, k_new, [0, 1, 2, 0], [16, 3, 0, -1],
                                   b.kv_indptr, b.kv_page_indices, P)
    assert skipped == 3
    page = int(b.kv_page_indices[b.kv_indptr[1]])
    assert torch.equal(k2[page, 3], k_new[1]) and torch.equal(v2[page, 3], k_new[1])
    changed = (k2 != b.k_cache.cpu()).any(dim=(1, 2, 3)).nonzero().flatten().tolist()
    assert changed == [page]
