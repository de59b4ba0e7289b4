"""Seeded random sweep over the decode path's parameters in combination.

Each case draws a batch size, request lengths (empty requests, very short
and long ones, ragged last pages), page size, head ratio, dtype, CTA budget,
minimum chunks per request, loader, page layout, softmax scale and logit
magnitude, and compares the whole batch with the oracle ("FlashInfer"
(aiwiki.ai/wiki/flashinfer), "Block-sparse / paged KV-cache", "Attention
states": paged decode, split work units, the LSE merge).  HND cases are also
checked bit-identical to the same data in NHD.  The cases are fixed by their
seeds, so a failure names a reproducible case.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

N_CASES = 240
MAX_TOKENS = 24000      # keeps the oracle at well under a second per case


def _case(i):
    rng = np.random.default_rng([7919, i])
    hkv = int(rng.choice([1, 2, 4, 8]))
    group = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16]))
    page = int(rng.choice([1, 2, 3, 5, 8, 16, 32, 64]))
    batch = int(rng.integers(1, 17))
    kind = int(rng.integers(0, 3))
    if kind == 0:      # short requests
        lengths = rng.integers(0, 300, batch)
    elif kind == 1:    # uniform, some long
        lengths = rng.integers(1, 3000, batch)
    else:              # heavy tail
        lengths = np.exp(rng.normal(math.log(300), 1.2, batch)).astype(np.int64)
    lengths = np.clip(lengths, 0, 8000)
    if rng.random() < 0.3:
        lengths[int(rng.integers(0, batch))] = 0
    if lengths.sum() > MAX_TOKENS:
        lengths = (lengths * (MAX_TOKENS / lengths.sum())).astype(np.int64)
    tma_ok = page % 16 == 0
    return dict(
        hkv=hkv, hq=hkv * group, page=page, lengths=[int(x) for x in lengths],
        dtype="f16" if rng.random() < 0.5 else "bf16",
        num_ctas=int(rng.choice([1, 5, 37, 152, 400])),
        min_chunks=int(rng.choice([1, 1, 2, 7])),
        loader=(pkd.LOADER_TMA_TILES if tma_ok and rng.random() < 0.3 else
                pkd.LOADER_BULK_ROWS if rng.random() < 0.2 else pkd.LOADER_AUTO),
        hnd=bool(rng.random() < 0.3),
        sm_scale=float(rng.choice([1.0 / math.sqrt(128), 0.05, 0.2])),
        k_scale=float(rng.choice([1.0, 0.25, 3.0])),
        spare_pages=int(rng.integers(0, 40)),
        seed=1000 + i)


def _run(wl, k, v, c, layout, loader):
    prob = pkd.make_problem(batch=wl.table.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=wl.table.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages, num_ctas=c["num_ctas"],
                            min_chunks_per_request=c["min_chunks"], kv_loader=loader,
                            kv_layout=layout)
    ws = pkd.Workspace(prob)
    plan = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, wl.table.kv_indices)
    out, lse = ws.run(plan, wl.q.cuda(), k, v, *gh.device_table(wl.table), c["sm_scale"])
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0
    return out, lse


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(i):
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    c = _case(i)
    used = sum((n + c["page"] - 1) // c["page"] for n in c["lengths"])
    wl = workloads.make_paged("sweep", c["lengths"], num_qo_heads=c["hq"],
                              num_kv_heads=c["hkv"], page_size=c["page"], dtype=c["dtype"],
                              seed=c["seed"], pool_pages=used + c["spare_pages"],
                              k_scale=c["k_scale"])
    ref_out, ref_lse = oracle.decode(
        workloads.as_codes(wl.q), workloads.as_codes(wl.k_pages),
        workloads.as_codes(wl.v_pages), wl.table.kv_indptr, wl.table.kv_indices,
        wl.table.kv_last_page_len, dtype=c["dtype"], sm_scale=c["sm_scale"])
    k, v = wl.k_pages.cuda(), wl.v_pages.cuda()
    loader_nhd = c["loader"]
    out, lse = _run(wl, k, v, c, pkd.LAYOUT_NHD, loader_nhd)
    gh.compare(out, lse, ref_out, ref_lse, c["dtype"])
    if c["hnd"]:
        k_hnd = k.transpose(1, 2).contiguous()
        v_hnd = v.transpose(1, 2).contiguous()
        out_h, lse_h = _run(wl, k_hnd, v_hnd, c, pkd.LAYOUT_HND, pkd.LOADER_AUTO)
        assert torch.equal(out_h, out) and torch.equal(lse_h, lse), c
