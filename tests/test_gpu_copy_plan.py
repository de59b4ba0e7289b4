"""pkd_copy_plan: a plan image copied from pinned host memory by a kernel.

"FlashInfer" (aiwiki.ai/wiki/flashinfer), "Plan and run": the host prepares
the schedule, and a captured run keeps its device addresses while the data
in them is updated.  The device copy must equal the host image byte for byte
(decode and shared-prefix plans); one captured graph [copy, decode, merge]
replayed after each new host plan written into the same pinned buffer must
match the oracle every time; an image larger than the workspace is refused on
the device (status word) without being copied past its header.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    pkd.load()


def _problem(wl, table, ctas, max_batch=0):
    return pkd.make_problem(batch=table.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=table.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=ctas,
                            max_batch=max_batch)


def test_device_copy_equals_host_image():
    wl = workloads.make_paged("copy", [3000, 17, 0, 900, 2500, 1], num_qo_heads=32,
                              num_kv_heads=8, page_size=16, dtype="f16", seed=5)
    for ctas in (1, 7, 152):
        ws = pkd.Workspace(_problem(wl, wl.table, ctas))
        ws.int_ws.fill_(0x5A)
        plan, img = pkd.plan_host(ws.problem, wl.table.kv_indptr, wl.table.kv_last_page_len,
                                  image=ws.staging[0])
        pkd.copy_plan(ws.staging[0], ws.int_ws)
        torch.cuda.synchronize()
        n = plan.int_ws_bytes_used
        dev = ws.int_ws[:n].cpu().numpy()
        host = ws.staging[0].numpy().view(np.uint8)[:n]
        assert np.array_equal(dev, host)
        # nothing past the plan's own words is written
        assert np.all(ws.int_ws[n:].cpu().numpy() == 0x5A)


def test_device_copy_of_prefix_image():
    prob = pkd.make_problem(batch=40, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=400, num_ctas=152)
    pws = pkd.PrefixWorkspace(prob, 300)
    pages = np.random.default_rng(1).permutation(400)[:190].astype(np.int32)
    plan, _ = pkd.plan_shared_prefix_host(prob, pages, 9, image=pws.staging)
    pkd.copy_plan(pws.staging, pws.int_ws)
    torch.cuda.synchronize()
    n = plan.int_ws_bytes_used
    assert np.array_equal(pws.int_ws[:n].cpu().numpy(),
                          pws.staging.numpy().view(np.uint8)[:n])


def test_captured_copy_follows_later_plans():
    """One graph [copy_plan, decode, merge] captured once at capacity 12,
    replayed after planning other batches into the same pinned buffer."""
    cap = 12
    rng = np.random.default_rng(7)
    lengths = rng.integers(1, 3000, size=cap)
    wl = workloads.make_paged("copy-graph", lengths, num_qo_heads=32, num_kv_heads=8,
                              page_size=16, dtype="bf16", seed=8)
    dev = gh.DeviceBatch(wl)
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    prob = _problem(wl, wl.table, ctas, max_batch=cap)
    ws = pkd.Workspace(prob)
    staging = ws.staging[0]
    # device page-table buffers sized for the capacity, refilled per plan
    nnz = int(wl.table.kv_indptr[-1])
    d_indptr = torch.zeros(cap + 1, dtype=torch.int32, device="cuda")
    d_indices = torch.zeros(max(nnz, 1), dtype=torch.int32, device="cuda")
    d_last = torch.zeros(cap, dtype=torch.int32, device="cuda")
    out = torch.zeros(cap, 32, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(cap, 32, dtype=torch.float32, device="cuda")

    def set_table(t):
        d_indptr[: t.batch + 1].copy_(torch.from_numpy(t.kv_indptr))
        if t.kv_indices.size:
            d_indices[: t.kv_indices.size].copy_(torch.from_numpy(t.kv_indices))
        d_last[: t.batch].copy_(torch.from_numpy(t.kv_last_page_len))

    plan, _ = pkd.plan_host(prob, wl.table.kv_indptr, wl.table.kv_last_page_len,
                            image=staging)
    set_table(wl.table)
    pkd.copy_plan(staging, ws.int_ws)
    ws.run(plan, dev.q, dev.k, dev.v, d_indptr, d_indices, d_last, wl.sm_scale,
           out=out, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkd.copy_plan(staging, ws.int_ws)
        ws.run(plan, dev.q, dev.k, dev.v, d_indptr, d_indices, d_last, wl.sm_scale,
               out=out, lse=lse)
    torch.cuda.synchronize()
    # later plans: sub-batches of the same requests (their pages stay put)
    for batch in (cap, 5, 1, 9):
        sel = list(range(batch))
        npages = np.diff(wl.table.kv_indptr.astype(np.int64))[sel]
        t = workloads.PageTable(
            np.concatenate([[0], np.cumsum(npages)]).astype(np.int32),
            wl.table.kv_indices[: int(npages.sum())].copy(),
            wl.table.kv_last_page_len[sel].copy(), 16)
        sub = _problem(wl, t, ctas, max_batch=cap)
        plan_b, _ = pkd.plan_host(sub, t.kv_indptr, t.kv_last_page_len, image=staging)
        set_table(t)
        g.replay()
        torch.cuda.synchronize()
        assert pkd.check_status(ws.int_ws) == 0
        ref_out, ref_lse = gh.oracle_ref(wl, table=t, q=wl.q[:batch].contiguous())
        gh.compare(out[:batch], lse[:batch], ref_out, ref_lse, "bf16")


def test_oversize_image_is_flagged_not_copied():
    wl = workloads.make_paged("copy-big", [4096] * 40, num_qo_heads=32, num_kv_heads=8,
                              page_size=1, dtype="f16", seed=9)
    ws = pkd.Workspace(_problem(wl, wl.table, 152))
    plan, _ = pkd.plan_host(ws.problem, wl.table.kv_indptr, wl.table.kv_last_page_len,
                            image=ws.staging[0])
    small = torch.full((plan.int_ws_bytes_used // 2,), 0x33, dtype=torch.uint8,
                       device="cuda")
    pkd.copy_plan(ws.staging[0], small)
    torch.cuda.synchronize()
    assert pkd.check_status(small) & pkd.DEVICE_BAD_PLAN
    assert np.all(small[64:].cpu().numpy() == 0x33)


def test_pageable_image_is_refused():
    ws_dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(1024, dtype=torch.int32)
    with pytest.raises(pkd.PkdError) as e:
        pkd.copy_plan(pageable, ws_dev)
    assert e.value.status == -1
