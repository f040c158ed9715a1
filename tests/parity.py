"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the fp64 oracle at the stated tolerances."""
import numpy as np
import torch

import paged_kv_decode_28_gb300 as pkd

# |gpu - oracle| <= ATOL_O + RTOL_O * |oracle| on outputs; |gpu - oracle| <= ATOL_LSE on lse
ATOL_O, RTOL_O, ATOL_LSE = 2e-3, 1e-2, 1e-3


def assert_o_close(got, ref, what="o"):
    g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    mask = ~np.isnan(ref)
    err = np.abs(g - ref)
    bound = ATOL_O + RTOL_O * np.abs(ref)
    bad = mask & ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(mask, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {mask.sum()} outside tolerance; worst at {i}: "
                             f"got {g[i]!r} want {ref[i]!r}")


def assert_lse_close(got, ref, what="lse"):
    g = got.detach().to("cpu", torch.float64).numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    mask = ~np.isnan(ref)
    both_ninf = np.isneginf(g) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_ninf, 0.0, np.abs(g - ref))
    bad = mask & ~(err <= ATOL_LSE)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(mask, np.nan_to_num(err, nan=np.inf), -np.inf)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {mask.sum()} outside tolerance; worst at {i}: "
                             f"got {g[i]!r} want {ref[i]!r}")


def to_device(batch, device="cuda"):
    return batch.to(device) if batch.q.device.type != "cuda" else batch


def gpu_paged_decode(batch, plan=None, check_errors=True):
    """Plan + run on the GPU for a workloads.PagedBatch (tensors moved to the GPU)."""
    b = to_device(batch)
    idx = torch.from_numpy(np.ascontiguousarray(b.kv_page_indices)).to("cuda")
    if plan is None:
        plan = pkd.Plan(max(b.batch, 1), b.num_qo_heads, b.num_kv_heads, b.head_dim)
    plan.plan(b.kv_indptr, idx, b.kv_last_page_len, b.page_size, q_dtype=b.q.dtype, kv_dtype=b.k_cache.dtype)
    out, lse = plan.run(b.q, b.k_cache, b.v_cache, sm_scale=b.sm_scale, k_scale=b.k_scale, v_scale=b.v_scale)
    torch.cuda.synchronize()
    if check_errors:
        assert plan.check_device_errors() == 0
    return out, lse, plan


def sample_rows(batch, n, seed=0):
    rng = np.random.default_rng(seed)
    B, Hq = batch.batch, batch.num_qo_heads
    rows = {(int(rng.integers(B)), int(rng.integers(Hq))) for _ in range(n)}
    # always include the longest request and the first / last heads
    longest = int(np.argmax(batch.kv_lens))
    rows |= {(longest, 0), (longest, Hq - 1), (B - 1, Hq - 1), (0, 0)}
    return sorted(rows)
