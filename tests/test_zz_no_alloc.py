"""pkd_run_static, the entry point that allocates no device memory.

It serves callers that cannot allocate device memory when they decode (their
device memory belongs to another allocator, or cudaMalloc's possible device
synchronisation is too costly in their loop): its scratch lives in a fixed
array inside the library.  Its output must match pkd_run's (the same kernels
with caller-allocated workspaces) on two calls in a row, the second over a
different batch, so stale contents of the shared array cannot leak into a
later call.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _batch(seed, lengths, dtype, hq):
    return workloads.make_paged("static%d" % seed, lengths, num_qo_heads=hq,
                                num_kv_heads=8, page_size=16, dtype=dtype, seed=seed)


def _static_run(dev, ctas):
    wl = dev.wl
    t = wl.table
    prob = pkd.make_problem(batch=t.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=t.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=ctas)
    plan, image = pkd.plan_host(prob, t.kv_indptr, t.kv_last_page_len, t.kv_indices)
    indptr, indices, last = gh.device_table(t)
    out, lse = pkd.run_static(plan, image, dev.q, dev.k, dev.v, indptr, indices, last,
                              wl.sm_scale)
    torch.cuda.synchronize()
    return out, lse, plan


def test_static_entry_matches_workspace_entry_twice():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    batches = [_batch(21, [3000, 17, 0, 900, 2500, 1], "f16", 32),
               _batch(22, [64, 4096, 333], "bf16", 64)]
    for wl in batches:
        dev = gh.DeviceBatch(wl)
        out_s, lse_s, plan = _static_run(dev, ctas)
        assert plan.num_split_requests > 0
        out_r, lse_r, _, _, status = gh.run_pkd(dev, num_ctas=ctas)
        assert status == 0
        ref_out = out_r.float().cpu().numpy().astype(np.float64).reshape(-1, 128)
        ref_lse = lse_r.cpu().numpy().astype(np.float64).reshape(-1)
        gh.compare(out_s, lse_s, ref_out, ref_lse, wl.dtype)


def test_static_entry_allocates_no_device_memory():
    """A warm call with caller-given out / lse leaves both torch's allocator
    and the device's free memory as they were."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    wl = _batch(23, [2000, 5, 700], "f16", 32)
    dev = gh.DeviceBatch(wl)
    t = wl.table
    prob = pkd.make_problem(batch=t.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=t.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=ctas)
    plan, image = pkd.plan_host(prob, t.kv_indptr, t.kv_last_page_len, t.kv_indices)
    assert plan.num_split_requests > 0
    indptr, indices, last = gh.device_table(t)
    out = torch.empty(t.batch, wl.num_qo_heads, 128, dtype=dev.q.dtype, device="cuda")
    lse = torch.empty(t.batch, wl.num_qo_heads, dtype=torch.float32, device="cuda")
    args = (plan, image, dev.q, dev.k, dev.v, indptr, indices, last, wl.sm_scale)
    pkd.run_static(*args, out=out, lse=lse)        # warm: address looked up
    torch.cuda.synchronize()
    first = out.clone(), lse.clone()
    torch.cuda.synchronize()
    allocated = torch.cuda.memory_allocated()
    free_before, _ = torch.cuda.mem_get_info()
    pkd.run_static(*args, out=out, lse=lse)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == allocated
    assert free_after == free_before
    assert torch.equal(out, first[0]) and torch.equal(lse, first[1])


def test_static_entry_rejects_short_host_image():
    prob = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=64, num_ctas=152)
    table = workloads.table_from_lengths([300, 40], 16, np.arange(64))
    plan, image = pkd.plan_host(prob, table.kv_indptr, table.kv_last_page_len)
    q = torch.empty(2, 32, 128, dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        pkd.run_static(plan, image[:-1], q, q, q, q, q, q, 0.1)


def test_static_entry_rejects_plans_beyond_its_limit():
    # 8 requests x 2000 pieces of 64 query heads: ~16 000 partial slots,
    # far beyond the 8 MiB of partial states the static array holds
    prob = pkd.make_problem(batch=8, num_qo_heads=64, num_kv_heads=8, page_size=16,
                            dtype="bf16", num_pages=1 << 20, num_ctas=152,
                            min_chunks_per_request=2000)
    table = workloads.table_from_lengths([32768] * 8, 16, np.arange(1 << 20))
    plan, image = pkd.plan_host(prob, table.kv_indptr, table.kv_last_page_len)
    assert plan.float_ws_bytes_needed > 8 * 1024 * 1024
    q = torch.empty(8, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkd.PkdError) as e:
        pkd.run_static(plan, image, q, q, q, q, q, q, 0.1)
    assert e.value.status == -3
    assert "static limit" in str(e.value)
