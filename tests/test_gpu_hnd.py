"""HND page layout ("Welcome to FlashInfer's documentation!", "KV-Cache Layout
in FlashInfer", "Layout: NHD/HND"): decode, shared prefix and append on HND
pools against the oracle, and decode bit-identical to the same data in NHD."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from oracle import append_ref
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _hnd(t):
    """[num_pages, P, Hkv, D] -> [num_pages, Hkv, P, D] (contiguous copy)."""
    return t.transpose(1, 2).contiguous()


def _run(wl, k, v, table, layout, loader=pkd.LOADER_AUTO, num_ctas=20):
    prob = pkd.make_problem(batch=table.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=table.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=num_ctas,
                            kv_loader=loader, kv_layout=layout)
    ws = pkd.Workspace(prob)
    plan = ws.plan(table.kv_indptr, table.kv_last_page_len, table.kv_indices)
    out, lse = ws.run(plan, wl.q.cuda(), k, v, *gh.device_table(table), wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0
    return out, lse


@pytest.mark.parametrize("page,dtype,hkv", [(16, "f16", 8), (64, "bf16", 8), (1, "bf16", 8),
                                            (5, "f16", 4), (32, "f16", 2)])
def test_hnd_decode(page, dtype, hkv):
    lengths = [0, 1, 70, 513, 16, 200]
    wl = workloads.make_paged("hnd", lengths, num_qo_heads=4 * hkv, num_kv_heads=hkv,
                              page_size=page, dtype=dtype, seed=page + hkv)
    k_nhd, v_nhd = wl.k_pages.cuda(), wl.v_pages.cuda()
    k_hnd, v_hnd = _hnd(k_nhd), _hnd(v_nhd)
    ref_out, ref_lse = oracle.decode(
        workloads.as_codes(wl.q), workloads.as_codes(_hnd(wl.k_pages)),
        workloads.as_codes(_hnd(wl.v_pages)), wl.table.kv_indptr, wl.table.kv_indices,
        wl.table.kv_last_page_len, dtype=dtype, sm_scale=wl.sm_scale, layout="HND")
    base = _run(wl, k_nhd, v_nhd, wl.table, pkd.LAYOUT_NHD)
    loaders = [pkd.LOADER_AUTO, pkd.LOADER_BULK_ROWS]
    if page % 16 == 0:
        loaders.append(pkd.LOADER_TMA_TILES)
    for loader in loaders:
        out, lse = _run(wl, k_hnd, v_hnd, wl.table, pkd.LAYOUT_HND, loader)
        gh.compare(out, lse, ref_out, ref_lse, dtype)
        assert torch.equal(out, base[0]) and torch.equal(lse, base[1])


def test_hnd_shared_prefix():
    batch, page, length = 12, 16, 777
    npages = (length + page - 1) // page
    wl = workloads.make_paged("hndp", [16] * batch, num_qo_heads=32, num_kv_heads=8,
                              page_size=page, dtype="bf16", seed=5, pool_pages=npages + batch)
    pages = np.random.default_rng(5).permutation(wl.num_pages)[:npages].astype(np.int32)
    last = length - (npages - 1) * page
    table = workloads.PageTable((np.arange(batch + 1) * npages).astype(np.int32),
                                np.tile(pages, batch), np.full(batch, last, np.int32), page)
    prob = pkd.make_problem(batch=batch, num_qo_heads=32, num_kv_heads=8, page_size=page,
                            dtype="bf16", num_pages=wl.num_pages, kv_layout=pkd.LAYOUT_HND)
    pws = pkd.PrefixWorkspace(prob, npages)
    plan = pws.plan(pages, last)
    out, lse = pws.run(plan, wl.q.cuda(), _hnd(wl.k_pages.cuda()), _hnd(wl.v_pages.cuda()),
                       wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(pws.int_ws) == 0
    ref_out, ref_lse = oracle.decode(
        workloads.as_codes(wl.q), workloads.as_codes(_hnd(wl.k_pages)),
        workloads.as_codes(_hnd(wl.v_pages)), table.kv_indptr, table.kv_indices,
        table.kv_last_page_len, dtype="bf16", sm_scale=wl.sm_scale, layout="HND")
    gh.compare(out, lse, ref_out, ref_lse, "bf16")


@pytest.mark.parametrize("page", [16, 3])
def test_hnd_append_is_bit_exact(page):
    lengths = [40, 7, 100]
    wl = workloads.make_paged("hnda", lengths, num_qo_heads=32, num_kv_heads=8,
                              page_size=page, dtype="f16", seed=page)
    t = wl.table
    rng = np.random.default_rng(page)
    bi = np.array([0, 0, 1, 2, 2, 2], np.int32)
    pos = np.array([39, 3, 6, 0, 55, 99], np.int32)
    kn = workloads._fill_normal((bi.size, 8, 128), "f16", 9, 5)
    vn = workloads._fill_normal((bi.size, 8, 128), "f16", 9, 6)
    k_hnd, v_hnd = _hnd(wl.k_pages), _hnd(wl.v_pages)
    k_ref, v_ref, skipped = append_ref.append_kv(
        workloads.as_codes(k_hnd), workloads.as_codes(v_hnd), workloads.as_codes(kn),
        workloads.as_codes(vn), bi, pos, t.kv_indptr, t.kv_indices, t.kv_last_page_len,
        layout="HND")
    assert skipped == []
    k_dev, v_dev = k_hnd.cuda(), v_hnd.cuda()
    prob = pkd.make_problem(batch=t.batch, num_qo_heads=32, num_kv_heads=8, page_size=page,
                            dtype="f16", num_pages=wl.num_pages, kv_layout=pkd.LAYOUT_HND)
    pkd.append_kv(prob, kn.cuda(), vn.cuda(), torch.from_numpy(bi).cuda(),
                  torch.from_numpy(pos).cuda(), k_dev, v_dev, *gh.device_table(t))
    torch.cuda.synchronize()
    assert np.array_equal(workloads.as_codes(k_dev.cpu()), k_ref)
    assert np.array_equal(workloads.as_codes(v_dev.cpu()), v_ref)
