"""A captured run stays valid for later plans ("FlashInfer"
(aiwiki.ai/wiki/flashinfer), "Plan and run": stable workspace addresses,
updated scheduling data passed to a captured run).

One CUDA graph holds the decode and merge launches; between replays the host
plans a different batch (other lengths, fewer requests, no split at all) into
the same workspace and rewrites the device page table in place.  Every replay
must match the oracle.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

MAX_BATCH = 6
POOL = 600


def _pool(dtype, seed):
    """A page pool and queries sized for MAX_BATCH requests."""
    return workloads.make_paged("graph", [16] * MAX_BATCH, num_qo_heads=32,
                                num_kv_heads=8, page_size=16, dtype=dtype, seed=seed,
                                pool_pages=POOL)


def _table(lengths, seed):
    perm = np.random.default_rng(seed).permutation(POOL)
    return workloads.table_from_lengths(lengths, 16, perm)


@pytest.mark.parametrize("dtype,loader", [("f16", pkd.LOADER_AUTO),
                                          ("bf16", pkd.LOADER_TMA_TILES)])
def test_captured_run_follows_later_plans(dtype, loader):
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    base = _pool(dtype, 40)
    dev = gh.DeviceBatch(base)
    prob = pkd.make_problem(batch=MAX_BATCH, num_qo_heads=32, num_kv_heads=8,
                            page_size=16, dtype=dtype, num_pages=POOL, num_ctas=24,
                            max_batch=MAX_BATCH, kv_loader=loader)
    ws = pkd.Workspace(prob)
    # device page table at fixed addresses, sized for the capacity
    indptr_d = torch.zeros(MAX_BATCH + 1, dtype=torch.int32, device="cuda")
    indices_d = torch.zeros(POOL, dtype=torch.int32, device="cuda")
    last_d = torch.zeros(MAX_BATCH, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(dev.q)
    lse = torch.zeros(dev.q.shape[:2], dtype=torch.float32, device="cuda")

    def load_table(t):
        indptr_d.zero_()
        last_d.zero_()
        indptr_d[: t.batch + 1].copy_(torch.from_numpy(t.kv_indptr))
        indices_d[: t.kv_indices.size].copy_(torch.from_numpy(t.kv_indices))
        last_d[: t.batch].copy_(torch.from_numpy(t.kv_last_page_len))

    first = _table([700, 33, 2000, 5, 1200, 64], 1)
    load_table(first)
    plan = ws.plan(first.kv_indptr, first.kv_last_page_len, first.kv_indices)
    assert plan.num_split_requests > 0
    # one eager run first (one-time per-device set-up happens outside capture)
    ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
           out=out, lse=lse)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
               out=out, lse=lse)

    cases = [first,
             _table([100, 2500, 17, 900, 0, 333], 2),   # other lengths
             _table([1500, 64, 700], 3),                # fewer requests
             _table([16, 3, 15, 1, 9, 12], 4)]          # nothing split
    for t in cases:
        load_table(t)
        p = ws.plan(t.kv_indptr, t.kv_last_page_len, t.kv_indices, batch=t.batch)
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert pkd.check_status(ws.int_ws) == 0
        wl = workloads.PagedBatch("graph", 32, 8, 128, dtype, base.q[: t.batch],
                                  base.k_pages, base.v_pages, t, base.sm_scale)
        ref_out, ref_lse = gh.oracle_ref(wl)
        gh.compare(out[: t.batch], lse[: t.batch], ref_out, ref_lse, dtype)
        if t is cases[-1]:
            assert p.num_split_requests == 0


def test_zero_requests():
    """A plan of no requests launches nothing eagerly and turns a captured
    decode + merge into a no-op; the graph then follows a non-empty plan."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    dtype = "f16"
    base = _pool(dtype, 41)
    dev = gh.DeviceBatch(base)
    empty = _table([], 5)

    # eager: PKD_OK, outputs untouched
    prob0 = pkd.make_problem(batch=0, num_qo_heads=32, num_kv_heads=8, page_size=16,
                             dtype=dtype, num_pages=POOL, num_ctas=24)
    ws0 = pkd.Workspace(prob0)
    plan0 = ws0.plan(empty.kv_indptr, empty.kv_last_page_len, empty.kv_indices)
    assert plan0.num_units == 0 and plan0.num_partials == 0
    out = torch.full_like(dev.q, 7.0)
    lse = torch.full(dev.q.shape[:2], 7.0, dtype=torch.float32, device="cuda")
    indptr0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws0.run(plan0, dev.q, dev.k, dev.v, indptr0, None, indptr0, base.sm_scale,
            out=out, lse=lse)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())

    # captured on a non-empty plan, replayed after an empty one, then a full one
    prob = pkd.make_problem(batch=MAX_BATCH, num_qo_heads=32, num_kv_heads=8,
                            page_size=16, dtype=dtype, num_pages=POOL, num_ctas=24,
                            max_batch=MAX_BATCH)
    ws = pkd.Workspace(prob)
    indptr_d = torch.zeros(MAX_BATCH + 1, dtype=torch.int32, device="cuda")
    indices_d = torch.zeros(POOL, dtype=torch.int32, device="cuda")
    last_d = torch.zeros(MAX_BATCH, dtype=torch.int32, device="cuda")

    def load_table(t):
        indptr_d.zero_()
        last_d.zero_()
        indptr_d[: t.batch + 1].copy_(torch.from_numpy(t.kv_indptr))
        indices_d[: t.kv_indices.size].copy_(torch.from_numpy(t.kv_indices))
        last_d[: t.batch].copy_(torch.from_numpy(t.kv_last_page_len))

    full = _table([900, 40, 1300, 7, 260, 2100], 6)
    load_table(full)
    plan = ws.plan(full.kv_indptr, full.kv_last_page_len, full.kv_indices)
    assert plan.num_split_requests > 0
    ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
           out=out, lse=lse)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
               out=out, lse=lse)

    load_table(empty)
    ws.plan(empty.kv_indptr, empty.kv_last_page_len, empty.kv_indices, batch=0)
    out.fill_(7.0)
    lse.fill_(7.0)
    graph.replay()
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0
    assert bool((out == 7.0).all()) and bool((lse == 7.0).all())

    load_table(full)
    ws.plan(full.kv_indptr, full.kv_last_page_len, full.kv_indices, batch=full.batch)
    graph.replay()
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0
    wl = workloads.PagedBatch("graph", 32, 8, 128, dtype, base.q[: full.batch],
                              base.k_pages, base.v_pages, full, base.sm_scale)
    ref_out, ref_lse = gh.oracle_ref(wl)
    gh.compare(out[: full.batch], lse[: full.batch], ref_out, ref_lse, dtype)


@pytest.mark.parametrize("seed", range(6))
def test_random_replays(seed):
    """One capture at a random capacity (max batch, CTAs, minimum chunks, page
    size, heads, dtype), replayed for five later plans of random batch and
    lengths (all-empty and tiny batches included); every replay against the
    oracle."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    rng = np.random.default_rng([5003, seed])
    max_batch = int(rng.integers(1, 13))
    page = int(rng.choice([1, 3, 16, 64]))
    hkv = int(rng.choice([1, 2, 8]))
    hq = hkv * int(rng.choice([1, 4, 5, 8]))
    dtype = "f16" if seed % 2 == 0 else "bf16"
    ctas = int(rng.choice([3, 40, 152]))
    m = int(rng.choice([1, 3]))
    max_len = 2500
    pool = max_batch * ((max_len + page - 1) // page) + 8
    base = workloads.make_paged("replay", [1] * max_batch, num_qo_heads=hq, num_kv_heads=hkv,
                                page_size=page, dtype=dtype, seed=seed + 50, pool_pages=pool)
    dev = gh.DeviceBatch(base)
    prob = pkd.make_problem(batch=max_batch, num_qo_heads=hq, num_kv_heads=hkv,
                            page_size=page, dtype=dtype, num_pages=pool, num_ctas=ctas,
                            min_chunks_per_request=m, max_batch=max_batch)
    ws = pkd.Workspace(prob)
    indptr_d = torch.zeros(max_batch + 1, dtype=torch.int32, device="cuda")
    indices_d = torch.zeros(pool, dtype=torch.int32, device="cuda")
    last_d = torch.zeros(max_batch, dtype=torch.int32, device="cuda")
    out = torch.zeros_like(dev.q)
    lse = torch.zeros(dev.q.shape[:2], dtype=torch.float32, device="cuda")

    def table(lengths):
        perm = rng.permutation(pool)
        return workloads.table_from_lengths(lengths, page, perm)

    def load_table(t):
        indptr_d.zero_()
        last_d.zero_()
        indptr_d[: t.batch + 1].copy_(torch.from_numpy(t.kv_indptr))
        if t.kv_indices.size:
            indices_d[: t.kv_indices.size].copy_(torch.from_numpy(t.kv_indices))
        if t.batch:
            last_d[: t.batch].copy_(torch.from_numpy(t.kv_last_page_len))

    first = table([int(x) for x in rng.integers(1, max_len, max_batch)])
    load_table(first)
    plan = ws.plan(first.kv_indptr, first.kv_last_page_len, first.kv_indices)
    ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
           out=out, lse=lse)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ws.run(plan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, base.sm_scale,
               out=out, lse=lse)

    later = [[int(x) for x in rng.integers(0, max_len, int(rng.integers(1, max_batch + 1)))]
             for _ in range(3)]
    later += [[0] * int(rng.integers(1, max_batch + 1)),                 # all empty
              [int(x) for x in rng.integers(1, 4, max_batch)]]          # tiny
    for lengths in later:
        t = table(lengths)
        load_table(t)
        ws.plan(t.kv_indptr, t.kv_last_page_len, t.kv_indices, batch=t.batch)
        out.zero_()
        lse.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert pkd.check_status(ws.int_ws) == 0, lengths
        wl = workloads.PagedBatch("replay", hq, hkv, 128, dtype, base.q[: t.batch],
                                  base.k_pages, base.v_pages, t, base.sm_scale)
        ref_out, ref_lse = gh.oracle_ref(wl)
        gh.compare(out[: t.batch], lse[: t.batch], ref_out, ref_lse, dtype)
