"""Shared-prefix (cascade) attention against the oracle.

"FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention states": a shared prefix
evaluated separately from the request-specific suffixes, then merged.  The
prefix kernel's states must equal attention over a table in which every
request lists the prefix pages; prefix states merged with suffix states must
equal attention over prefix + suffix.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from oracle import prefix_plan_ref
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _prefix_case(batch, hq, hkv, page, length, dtype, seed):
    npages = (length + page - 1) // page
    pool = max(npages, batch) + 5
    wl = workloads.make_paged("prefix", [16] * batch, num_qo_heads=hq, num_kv_heads=hkv,
                              page_size=page, dtype=dtype, seed=seed, pool_pages=pool)
    pages = np.random.default_rng(seed).permutation(pool)[:npages].astype(np.int32)
    last = length - (npages - 1) * page if npages else 0
    table = workloads.PageTable(
        (np.arange(batch + 1) * npages).astype(np.int32),
        np.tile(pages, batch).astype(np.int32),
        np.full(batch, last, dtype=np.int32), page)
    return wl, pages, last, table


def _run_prefix(dev, wl, pages, last, num_ctas=0):
    prob = pkd.make_problem(batch=wl.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=wl.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=num_ctas)
    pws = pkd.PrefixWorkspace(prob, max(1, pages.size))
    plan = pws.plan(pages, last)
    out, lse = pws.run(plan, dev.q, dev.k, dev.v, wl.sm_scale)
    torch.cuda.synchronize()
    return out, lse, plan, pkd.check_status(pws.int_ws)


CASES = [
    # batch, hq, hkv, page, prefix length, dtype, num_ctas
    (1, 32, 8, 16, 512, "f16", 0),
    (3, 32, 8, 16, 17, "bf16", 0),
    (40, 32, 8, 16, 3000, "f16", 0),
    (40, 32, 8, 16, 3000, "bf16", 7),
    (5, 64, 8, 64, 1000, "bf16", 0),
    (9, 8, 8, 32, 65, "f16", 152),
    (2, 16, 1, 16, 2049, "bf16", 3),
    (70, 32, 4, 16, 640, "f16", 0),
    (4, 32, 8, 16, 1, "f16", 0),
]


@pytest.mark.parametrize("case", CASES)
def test_shared_prefix_matches_oracle(case):
    batch, hq, hkv, page, length, dtype, ctas = case
    wl, pages, last, table = _prefix_case(batch, hq, hkv, page, length, dtype,
                                          seed=batch * 7 + length)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, status = _run_prefix(dev, wl, pages, last, ctas)
    assert status == 0
    assert plan.prefix_len == length and plan.chunks >= 1
    ref_out, ref_lse = gh.oracle_ref(wl, table=table)
    gh.compare(out, lse, ref_out, ref_lse, dtype)


@pytest.mark.parametrize("case", CASES)
def test_device_prefix_image_matches_restatement(case):
    """The image pkd_plan_shared_prefix copies to the device equals, byte for
    byte, the plain-Python restatement of the prefix planning rule."""
    batch, hq, hkv, page, length, dtype, ctas = case
    wl, pages, last, _ = _prefix_case(batch, hq, hkv, page, length, dtype,
                                      seed=batch * 7 + length)
    prob = pkd.make_problem(batch=wl.batch, num_qo_heads=hq, num_kv_heads=hkv,
                            page_size=page, dtype=dtype, num_pages=wl.num_pages,
                            num_ctas=ctas)
    pws = pkd.PrefixWorkspace(prob, max(1, pages.size))
    plan = pws.plan(pages, last)
    torch.cuda.synchronize()
    img = pws.int_ws[: plan.int_ws_bytes_used].cpu().numpy().view(np.int32)
    num_ctas = ctas or torch.cuda.get_device_properties(0).multi_processor_count
    scalars, ref_img = prefix_plan_ref.plan(batch, hq, hkv, page, pages, last, num_ctas)
    assert img.tobytes() == ref_img.tobytes()
    for key, value in scalars.items():
        assert getattr(plan, key) == value, key


def test_shared_prefix_rejects_bad_pages_and_page_sizes():
    wl, pages, last, _ = _prefix_case(2, 32, 8, 16, 100, "f16", 1)
    prob = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=wl.num_pages, num_ctas=8)
    pws = pkd.PrefixWorkspace(prob, 16)
    bad = pages.copy()
    bad[1] = wl.num_pages
    with pytest.raises(pkd.PkdError) as e:
        pws.plan(bad, last)
    assert e.value.status == -2
    with pytest.raises(pkd.PkdError) as e:
        pws.plan(pages, 17)
    assert e.value.status == -2
    prob8 = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=8,
                             dtype="f16", num_pages=100, num_ctas=8)
    with pytest.raises(pkd.PkdError) as e:
        pkd.PrefixWorkspace(prob8, 16).plan(np.arange(3, dtype=np.int32), 8)
    assert e.value.status == -4


def test_cascade_shared_prefix_plus_suffix():
    wl = workloads.cascade()
    dev = gh.DeviceBatch(wl)
    prefix = wl.extra_tables["prefix"]
    pages = prefix.kv_indices[: prefix.kv_indptr[1]]
    pre_out, pre_lse, plan, st1 = _run_prefix(dev, wl, pages,
                                              int(prefix.kv_last_page_len[0]))
    suf_out, suf_lse, _, _, st2 = gh.run_pkd(dev, wl.extra_tables["suffix"])
    assert st1 == 0 and st2 == 0
    out, lse = pkd.merge_states(pre_out, pre_lse, suf_out, suf_lse)
    torch.cuda.synchronize()
    rng = np.random.default_rng(8)
    total = wl.batch * wl.num_qo_heads
    rows = np.unique(np.concatenate([rng.choice(total, 300, replace=False),
                                     [0, total - 1]])).astype(np.int64)
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)
    print("cascade (shared prefix)", plan.chunks, plan.row_tiles,
          gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows))


@pytest.mark.parametrize("dtype,length,ctas", [("f16", 3000, 8), ("bf16", 1500, 4),
                                               ("f16", 700, 152)])
def test_shared_prefix_growing_scores(dtype, length, ctas):
    # keys grow along the prefix, so the running maximum keeps rising and the
    # reference moves (rescaling the accumulated output) after the first tile
    batch = 6
    wl, pages, last, table = _prefix_case(batch, 32, 8, 16, length, dtype, seed=length)
    k = wl.k_pages.float()
    for t in range(length):
        k[pages[t // 16], t % 16] *= 1.0 + 7.0 * t / length
    wl.k_pages = k.to(wl.k_pages.dtype)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, status = _run_prefix(dev, wl, pages, last, ctas)
    assert status == 0
    ref_out, ref_lse = gh.oracle_ref(wl, table=table)
    gh.compare(out, lse, ref_out, ref_lse, dtype)
    # the last tokens dominate: the growth really moved the maximum
    assert float(ref_lse.max()) > 8.0


def test_shared_prefix_empty():
    wl, _, _, _ = _prefix_case(3, 32, 8, 16, 16, "f16", seed=5)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, status = _run_prefix(dev, wl, np.zeros(0, np.int32), 0)
    assert status == 0 and plan.prefix_len == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_shared_prefix_single_dominant_token(dtype):
    # one prefix key points along query row (request 0, head 0): that row's
    # weights collapse onto a single token, so its output is one value row and
    # any mismatch between the normaliser and the rounded weights shows
    batch, length = 4, 700
    wl, pages, last, table = _prefix_case(batch, 32, 8, 16, length, dtype, seed=41)
    q0 = wl.q[0, 0].float()
    k = wl.k_pages.float()
    v = wl.v_pages.float()
    t_star = 333
    k[pages[t_star // 16], t_star % 16, 0] = q0 * (4.0 / q0.norm()) * (128 ** 0.5)
    v[pages[t_star // 16], t_star % 16, 0] = torch.linspace(-4.5, 4.5, 128)
    wl.k_pages = k.to(wl.k_pages.dtype)
    wl.v_pages = v.to(wl.v_pages.dtype)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, status = _run_prefix(dev, wl, pages, last, 8)
    assert status == 0
    ref_out, ref_lse = gh.oracle_ref(wl, table=table)
    gh.compare(out, lse, ref_out, ref_lse, dtype)
    # the row really is dominated by that token
    v_star = wl.v_pages[pages[t_star // 16], t_star % 16, 0].float().numpy()
    assert np.abs(ref_out[0] - v_star).max() < 1e-3
