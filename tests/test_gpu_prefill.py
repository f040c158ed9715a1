"""GPU parity of paged prefill / append attention (several query tokens per
request, the causal mask aligned to the end of each sequence) on the
tile-attention kernel, against the oracle: ragged query and key counts that
span several 128-row and 128-key tiles, causal and not, page sizes, group
sizes, f16/bf16, HND pools, a full-sequence prefill, the append-then-prefill
flow, a serving-size batch with sampled rows, and argument checks."""
import numpy as np
import pytest
import torch

import paged_kv_decode_28_gb300 as pkd
from oracle import attention as orc
from oracle import kv_append as ka
from paged_kv_decode_28_gb300 import workloads as wl
from tests.parity import assert_lse_close, assert_o_close

pytestmark = pytest.mark.gpu


def _cuda_i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()


def _gpu_prefill(b, causal=True, layout="NHD", kc=None, vc=None):
    plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads, kv_layout=layout)
    plan.plan_prefill(b.qo_indptr, b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, b.page_size,
                      causal=causal, q_dtype=b.q.dtype)
    out, lse = plan.prefill(b.q, b.k_cache if kc is None else kc, b.v_cache if vc is None else vc,
                            sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert plan.check_device_errors() == 0
    return out, lse


def _oracle(b, causal=True, rows=None):
    return orc.paged_prefill(b.q, b.qo_indptr, b.k_cache, b.v_cache, b.kv_indptr, b.kv_page_indices,
                             b.kv_last_page_len, causal=causal, sm_scale=b.sm_scale, rows=rows)


Q_LENS = [1, 0, 31, 32, 33, 100, 7, 250]
KV_LENS = [1, 5, 31, 160, 33, 300, 1000, 250]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("P", [1, 16, 64, 128])
@pytest.mark.parametrize("g", [1, 4, 8])
def test_prefill_matches_oracle(causal, P, g):
    b = wl.make_prefill(seed=1200 + P + g, q_lens=Q_LENS, kv_lens=KV_LENS, num_qo_heads=2 * g, num_kv_heads=2,
                        page_size=P, device="cuda")
    out, lse = _gpu_prefill(b, causal)
    o_ref, l_ref = _oracle(b, causal)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


@pytest.mark.parametrize("g", [1, 4])
def test_lone_tiles_split_over_key_tiles(g):
    """A request's lone last query tile with two or more key tiles takes its
    even and odd key tiles in two halves and combines them: rows that see no
    key of the odd tiles (causal rows before key 128), three key tiles, a tile
    cut by the sequence end."""
    b = wl.make_prefill(seed=1240 + g, q_lens=[100, 20, 3, 30, 1], kv_lens=[150, 140, 300, 140, 257],
                        num_qo_heads=2 * g, num_kv_heads=2, page_size=16, device="cuda")
    for causal in (True, False):
        out, lse = _gpu_prefill(b, causal)
        o_ref, l_ref = _oracle(b, causal)
        assert_o_close(out, o_ref, what=f"causal={causal}")
        assert_lse_close(lse, l_ref, what=f"causal={causal}")


def test_prefill_growing_scores():
    """Keys whose norm grows page by page along each sequence, so a row's
    running maximum rises by more than the lazy-rescale threshold many times
    over its key tiles (O rescaled in TMEM between products), causal and not,
    bf16 and f16."""
    for dt in ("bf16", "f16"):
        b = wl.make_prefill(seed=1290, q_lens=[40, 130, 7, 256], kv_lens=[700, 520, 900, 300], num_qo_heads=8,
                            num_kv_heads=2, page_size=16, q_dtype=dt, kv_dtype=dt, device="cuda")
        ip = b.kv_indptr
        for r in range(len(ip) - 1):
            for pos, pid in enumerate(b.kv_page_indices[ip[r]:ip[r + 1]].tolist()):
                b.k_cache[pid] *= 1.0 + 0.25 * pos
        for causal in (True, False):
            out, lse = _gpu_prefill(b, causal)
            o_ref, l_ref = _oracle(b, causal)
            assert_o_close(out, o_ref, what=f"{dt} causal={causal}")
            assert_lse_close(lse, l_ref, what=f"{dt} causal={causal}")


def test_prefill_f16_and_hnd():
    from tests.test_gpu_hnd import to_hnd

    b = wl.make_prefill(seed=1250, q_lens=Q_LENS, kv_lens=KV_LENS, num_qo_heads=16, num_kv_heads=4, page_size=16,
                        q_dtype="f16", kv_dtype="f16", device="cuda")
    out, lse = _gpu_prefill(b)
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)
    out_h, lse_h = _gpu_prefill(b, layout="HND", kc=to_hnd(b.k_cache), vc=to_hnd(b.v_cache))
    assert torch.equal(out_h, out) and torch.equal(lse_h, lse)


def test_full_sequence_prefill():
    """q_len == kv_len: every token of a 1000-token prompt attends its prefix."""
    b = wl.make_prefill(seed=1260, q_lens=[1000, 129], kv_lens=[1000, 129], num_qo_heads=32, num_kv_heads=8,
                        page_size=16, device="cuda")
    out, lse = _gpu_prefill(b)
    rng = np.random.default_rng(0)
    rows = sorted({(int(t), int(h)) for t, h in zip(rng.integers(0, 1129, 200), rng.integers(0, 32, 200))} |
                  {(0, 0), (999, 31), (1000, 5), (1128, 0)})
    o_ref, l_ref = _oracle(b, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_append_then_prefill():
    """The append flow: new tokens' K/V are written into their pages with
    pkd_append_kv, then their queries attend the whole cache causally."""
    old, new = np.array([40, 0, 300, 17]), np.array([16, 9, 64, 1])
    b = wl.make_prefill(seed=1270, q_lens=new, kv_lens=old + new, num_qo_heads=16, num_kv_heads=4, page_size=16,
                        device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(3)
    T = int(new.sum())
    k_new = torch.randn(T, 4, 128, device="cuda", generator=gen).to(torch.bfloat16)
    v_new = torch.randn(T, 4, 128, device="cuda", generator=gen).to(torch.bfloat16)
    bi = np.repeat(np.arange(len(new)), new)
    pos = np.concatenate([np.arange(o, o + n) for o, n in zip(old, new)])
    kr, vr, skipped = ka.append_kv(b.k_cache, b.v_cache, k_new, v_new, bi, pos, b.kv_indptr, b.kv_page_indices, 16)
    assert skipped == 0
    pkd.append_kv(k_new, v_new, _cuda_i32(bi), _cuda_i32(pos), _cuda_i32(b.kv_indptr),
                  _cuda_i32(b.kv_page_indices), b.k_cache, b.v_cache)
    out, lse = _gpu_prefill(b)  # ordered after the append on the stream
    b.k_cache, b.v_cache = kr, vr
    o_ref, l_ref = _oracle(b)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_prefill_serving_size_sampled():
    b = wl.make_config_prefill(device="cuda")
    out, lse = _gpu_prefill(b)
    rng = np.random.default_rng(1)
    T = b.q.shape[0]
    rows = sorted({(int(t), int(h)) for t, h in zip(rng.integers(0, T, 64), rng.integers(0, b.num_qo_heads, 64))}
                  | {(int(t) - 1, 0) for t in b.qo_indptr[1:]})
    o_ref, l_ref = _oracle(b, rows=rows)
    assert_o_close(out, o_ref)
    assert_lse_close(lse, l_ref)


def test_prefill_bad_arguments():
    b = wl.make_prefill(seed=1280, q_lens=[4], kv_lens=[4], num_qo_heads=8, num_kv_heads=2, page_size=16,
                        device="cuda")
    plan = pkd.Plan(1, 8, 2)
    with pytest.raises(pkd.PkdError):  # more query tokens than keys
        plan.plan_prefill([0, 5], b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, 16)
    with pytest.raises(pkd.PkdError):  # prefill before a prefill plan
        plan.prefill(b.q, b.k_cache, b.v_cache)
    with pytest.raises(pkd.PkdError):  # e4m3 K/V is not built for prefill
        plan.plan_prefill(b.qo_indptr, b.kv_indptr, _cuda_i32(b.kv_page_indices), b.kv_last_page_len, 16,
                          kv_dtype=torch.float8_e4m3fn)
