"""Cascade attention in one call (pkd_run_cascade) against the oracle.

"FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention states": the state of a
shared prefix and the state of a request's own suffix merge into the state
over both.  The reference is the oracle's attention over the prefix table
and over the suffix table, merged by the oracle's merge (pinned on its own
by the union tests), so prefixes need not fill whole pages.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _case(batch, hq, hkv, page, prefix_len, suffix_lens, dtype, seed):
    """Queries and a pool holding a shared prefix and per-request suffixes."""
    npre = (prefix_len + page - 1) // page
    nsuf = sum((n + page - 1) // page for n in suffix_lens)
    pool = npre + nsuf + 3
    wl = workloads.make_paged("cascade-case", [16] * batch, num_qo_heads=hq,
                              num_kv_heads=hkv, page_size=page, dtype=dtype, seed=seed,
                              pool_pages=pool)
    perm = np.random.default_rng(seed).permutation(pool).astype(np.int32)
    pre_pages = perm[:npre]
    pre_last = prefix_len - (npre - 1) * page if npre else 0
    prefix = workloads.PageTable((np.arange(batch + 1) * npre).astype(np.int32),
                                 np.tile(pre_pages, batch).astype(np.int32),
                                 np.full(batch, pre_last, dtype=np.int32), page)
    suffix = workloads.table_from_lengths(list(suffix_lens), page, perm[npre:npre + nsuf])
    return wl, pre_pages, pre_last, prefix, suffix


def _reference(wl, prefix, suffix):
    po, ps = gh.oracle_ref(wl, table=prefix)
    so, ss = gh.oracle_ref(wl, table=suffix)
    return oracle.merge(po, ps, so, ss)


def _setup(wl, pre_pages, pre_last, suffix, num_ctas, min_chunks, layout=pkd.LAYOUT_NHD):
    prob = pkd.make_problem(batch=wl.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=wl.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=num_ctas,
                            min_chunks_per_request=min_chunks, kv_layout=layout)
    ws = pkd.Workspace(prob)
    plan = ws.plan(suffix.kv_indptr, suffix.kv_last_page_len, suffix.kv_indices)
    pws = pkd.PrefixWorkspace(prob, max(1, pre_pages.size))
    pplan = pws.plan(pre_pages, pre_last)
    return ws, plan, pws, pplan


CASES = [
    # batch, hq, hkv, page, prefix length, suffix lengths, dtype, num_ctas, min_chunks
    (5, 32, 8, 16, 700, [0, 1, 50, 600, 2000], "f16", 0, 1),
    (5, 32, 8, 16, 700, [0, 1, 50, 600, 2000], "bf16", 8, 1),
    (3, 64, 8, 16, 129, [300, 0, 17], "bf16", 0, 4),
    (4, 32, 8, 32, 0, [100, 0, 64, 33], "f16", 0, 1),
    (4, 32, 8, 16, 1000, [0, 0, 0, 0], "f16", 0, 1),
    (2, 16, 1, 16, 2049, [500, 1000], "bf16", 3, 2),
    (33, 32, 4, 16, 64, list(range(1, 33 * 37, 37)), "f16", 0, 1),
]


@pytest.mark.parametrize("case", CASES)
def test_cascade_matches_oracle(case):
    batch, hq, hkv, page, plen, slens, dtype, ctas, m = case
    wl, pre_pages, pre_last, prefix, suffix = _case(batch, hq, hkv, page, plen, slens,
                                                    dtype, seed=7 * batch + plen)
    dev = gh.DeviceBatch(wl)
    ws, plan, pws, pplan = _setup(wl, pre_pages, pre_last, suffix, ctas, m)
    indptr, indices, last = gh.device_table(suffix)
    out, lse = pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr, indices, last,
                               ws, pws, wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0 and pkd.check_status(pws.int_ws) == 0
    ref_out, ref_lse = _reference(wl, prefix, suffix)
    gh.compare(out, lse, ref_out, ref_lse, dtype)


def test_cascade_pieces_equal_the_single_call():
    # prefix states, suffix decode and the cascade merge launched one by one
    # give the single call's bits
    wl, pre_pages, pre_last, prefix, suffix = _case(6, 32, 8, 16, 900,
                                                    [40, 0, 3000, 7, 800, 1500], "bf16", 5)
    dev = gh.DeviceBatch(wl)
    ws, plan, pws, pplan = _setup(wl, pre_pages, pre_last, suffix, 16, 1)
    assert plan.num_split_requests > 0
    indptr, indices, last = gh.device_table(suffix)
    one, one_lse = pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr, indices, last,
                                   ws, pws, wl.sm_scale)
    pws.run_states(pplan, dev.q, dev.k, dev.v, wl.sm_scale)
    ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, wl.sm_scale,
           phase="decode_states")
    out, lse = torch.empty_like(one), torch.empty_like(one_lse)
    pkd.run_cascade_merge(plan, pplan, ws, pws, out, lse)
    torch.cuda.synchronize()
    assert torch.equal(out, one) and torch.equal(lse, one_lse)
    gh.compare(out, lse, *_reference(wl, prefix, suffix), "bf16")


def test_cascade_rejects_mismatched_plans():
    wl, pre_pages, pre_last, _, suffix = _case(3, 32, 8, 16, 100, [10, 20, 30], "f16", 9)
    dev = gh.DeviceBatch(wl)
    ws, plan, _, _ = _setup(wl, pre_pages, pre_last, suffix, 0, 1)
    other = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=16,
                             dtype="f16", num_pages=wl.num_pages)
    pws = pkd.PrefixWorkspace(other, 16)
    pplan = pws.plan(pre_pages, pre_last)
    indptr, indices, last = gh.device_table(suffix)
    out = torch.full_like(dev.q, 7.0)
    lse = torch.zeros(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    with pytest.raises(pkd.PkdError) as e:
        pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr, indices, last, ws, pws,
                        wl.sm_scale, out=out, lse=lse)
    assert e.value.status == -1
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)  # nothing launched


def test_cascade_workload_sampled_rows():
    wl = workloads.cascade()
    dev = gh.DeviceBatch(wl)
    pt, st = wl.extra_tables["prefix"], wl.extra_tables["suffix"]
    pre_pages = pt.kv_indices[: pt.kv_indptr[1]].copy()
    ws, plan, pws, pplan = _setup(wl, pre_pages, int(pt.kv_last_page_len[0]), st, 0, 1)
    indptr, indices, last = gh.device_table(st)
    out, lse = pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr, indices, last,
                               ws, pws, wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0 and pkd.check_status(pws.int_ws) == 0
    total = wl.batch * wl.num_qo_heads
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([rng.choice(total, 300, replace=False),
                                     [0, total - 1]])).astype(np.int64)
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)   # the combined prefix + suffix table
    print("cascade (one call)", pplan.chunks, plan.num_split_requests,
          gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows))


def test_captured_cascade_follows_later_suffix_plans():
    batch = 5
    wl, pre_pages, pre_last, prefix, first = _case(batch, 32, 8, 16, 1100,
                                                   [700, 0, 2000, 5, 1200], "f16", 21)
    dev = gh.DeviceBatch(wl)
    ws, plan, pws, pplan = _setup(wl, pre_pages, pre_last, first, 20, 1)
    assert plan.num_split_requests > 0
    npages = wl.num_pages
    indptr_d = torch.zeros(batch + 1, dtype=torch.int32, device="cuda")
    indices_d = torch.zeros(npages, dtype=torch.int32, device="cuda")
    last_d = torch.zeros(batch, dtype=torch.int32, device="cuda")

    def load_table(t):
        indptr_d.copy_(torch.from_numpy(t.kv_indptr))
        indices_d.zero_()
        indices_d[: t.kv_indices.size].copy_(torch.from_numpy(t.kv_indices))
        last_d.copy_(torch.from_numpy(t.kv_last_page_len))

    out = torch.zeros_like(dev.q)
    lse = torch.zeros(dev.q.shape[:2], dtype=torch.float32, device="cuda")
    load_table(first)
    pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, ws, pws,
                    wl.sm_scale, out=out, lse=lse)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, indptr_d, indices_d, last_d, ws,
                        pws, wl.sm_scale, out=out, lse=lse)
    # later suffix tables over the suffix part of the pool (the prefix pages
    # are not reused), the same batch
    free = np.setdiff1d(np.arange(npages, dtype=np.int32), pre_pages)
    later = [first,
             workloads.table_from_lengths([100, 1500, 17, 0, 333], 16,
                                          np.random.default_rng(2).permutation(free)),
             workloads.table_from_lengths([16, 3, 15, 1, 9], 16,
                                          np.random.default_rng(3).permutation(free))]
    for t in later:
        load_table(t)
        ws.plan(t.kv_indptr, t.kv_last_page_len, t.kv_indices)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert pkd.check_status(ws.int_ws) == 0 and pkd.check_status(pws.int_ws) == 0
        gh.compare(out, lse, *_reference(wl, prefix, t), "f16")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_cascade_hnd_pages_equal_nhd(dtype):
    # the same values in [pages][Hkv][P][D]: the same bits as the NHD run
    wl, pre_pages, pre_last, prefix, suffix = _case(4, 32, 8, 16, 600, [30, 900, 0, 2500],
                                                    dtype, 13)
    dev = gh.DeviceBatch(wl)
    indptr, indices, last = gh.device_table(suffix)
    results = []
    for layout in (pkd.LAYOUT_NHD, pkd.LAYOUT_HND):
        k, v = dev.k, dev.v
        if layout == pkd.LAYOUT_HND:
            k, v = k.transpose(1, 2).contiguous(), v.transpose(1, 2).contiguous()
        ws, plan, pws, pplan = _setup(wl, pre_pages, pre_last, suffix, 12, 1, layout)
        out, lse = pkd.run_cascade(plan, pplan, dev.q, k, v, indptr, indices, last, ws, pws,
                                   wl.sm_scale)
        torch.cuda.synchronize()
        assert pkd.check_status(ws.int_ws) == 0 and pkd.check_status(pws.int_ws) == 0
        results.append((out, lse))
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])
    gh.compare(results[1][0], results[1][1], *_reference(wl, prefix, suffix), dtype)


def _random_case(i):
    """Seeded draw: batch, heads (any group up to 16, so the prefix kernel's
    plain query loads for 128 % g != 0 are covered), page size, prefix and
    suffix lengths (empty ones included), dtype, CTA budget, chunks."""
    rng = np.random.default_rng([4241, i])
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16]))
    batch = int(rng.integers(1, 41))
    prefix_len = int(rng.choice([0, 1, int(rng.integers(2, 200)), int(rng.integers(200, 4000))]))
    suffix = rng.integers(0, 2000, batch)
    suffix[rng.random(batch) < 0.15] = 0
    return dict(batch=batch, hq=hkv * group, hkv=hkv, page=int(rng.choice([16, 32, 64])),
                prefix_len=prefix_len, suffix=[int(x) for x in suffix],
                dtype="f16" if rng.random() < 0.5 else "bf16",
                num_ctas=int(rng.choice([0, 5, 37, 152])),
                min_chunks=int(rng.choice([1, 2, 4])), seed=300 + i)


@pytest.mark.parametrize("i", range(64))
def test_cascade_random_cases(i):
    c = _random_case(i)
    wl, pre_pages, pre_last, prefix, suffix = _case(c["batch"], c["hq"], c["hkv"], c["page"],
                                                    c["prefix_len"], c["suffix"], c["dtype"],
                                                    c["seed"])
    dev = gh.DeviceBatch(wl)
    ws, plan, pws, pplan = _setup(wl, pre_pages, pre_last, suffix, c["num_ctas"],
                                  c["min_chunks"])
    out, lse = pkd.run_cascade(plan, pplan, dev.q, dev.k, dev.v, *gh.device_table(suffix),
                               ws, pws, wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0 and pkd.check_status(pws.int_ws) == 0
    gh.compare(out, lse, *_reference(wl, prefix, suffix), c["dtype"])
