"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case compares element by element on the same seeded inputs; the bounds
are in tests/gpu_helpers.py.  Cases: the adversarial kinds the pages list
(tests/golden/adversarial_cases.json), the five measured workloads (all rows
where the oracle finishes in seconds, sampled rows otherwise, in the launch
configuration the benchmark times), several split geometries for one batch,
the cascade (prefix and suffix runs merged with merge_states), plan reuse and
the device-side range checks.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from oracle import plan_ref
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CASES = json.load(open(os.path.join(HERE, "golden", "adversarial_cases.json")))["cases"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    pkd.load()


def _codes(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        workloads.TORCH_DTYPES[dtype])


def build_case(case, seed=99):
    wl = workloads.make_paged(case["name"], case["lengths"],
                              num_qo_heads=case["num_qo_heads"],
                              num_kv_heads=case["num_kv_heads"],
                              page_size=case["page_size"], dtype=case["dtype"],
                              seed=seed, pool_pages=None)
    extreme = case.get("extreme")
    if extreme:
        rng = np.random.default_rng(seed)
        halves = np.array([-1.0, -0.5, 0.0, 0.5, 1.0], dtype=np.float32)
        q = rng.choice(halves, size=tuple(wl.q.shape))
        k = rng.choice(halves, size=tuple(wl.k_pages.shape))
        if extreme == "negative":
            # every raw dot product is -2^20 + (multiple of 1/4, |.| <= 127):
            # exact in fp32, all logits near -9.3e4
            q[..., 0] = 1024.0
            k[..., 0] = -1024.0
        else:
            q[..., 0] = 256.0
            k[..., 0] = rng.integers(-64, 65, size=k.shape[:-1])
        wl.q = _codes(q, wl.dtype)
        wl.k_pages = _codes(k, wl.dtype)
    return wl


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_adversarial_case(case):
    wl = build_case(case)
    dev = gh.DeviceBatch(wl)
    for num_ctas, m in ((0, 1), (3, 4)):
        out, lse, plan, ws, status = gh.run_pkd(dev, num_ctas=num_ctas, min_chunks=m)
        assert status == 0
        ref_out, ref_lse = gh.oracle_ref(wl)
        if case.get("extreme") == "negative":
            assert np.all(ref_lse[np.isfinite(ref_lse)] < -5e4)
        gh.compare(out, lse, ref_out, ref_lse, wl.dtype)


def _workload(name):
    return workloads.WORKLOADS[name]()


@pytest.mark.parametrize("name", ["single", "batch64", "longtail"])
def test_workload_all_rows(name):
    wl = _workload(name)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, ws, status = gh.run_pkd(dev)
    assert status == 0
    ref_out, ref_lse = gh.oracle_ref(wl)
    summary = gh.compare(out, lse, ref_out, ref_lse, wl.dtype)
    print(name, summary, "units", plan.num_units, "split", plan.num_split_requests)


def _sample_rows(wl, n, seed):
    rng = np.random.default_rng(seed)
    total = wl.batch * wl.num_qo_heads
    rows = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    rows.update([0, total - 1, wl.num_qo_heads - 1])
    return np.array(sorted(rows), dtype=np.int64)


def test_longctx_sampled_rows():
    wl = _workload("longctx")
    dev = gh.DeviceBatch(wl)
    out, lse, plan, ws, status = gh.run_pkd(dev)
    assert status == 0
    # the per-request reading of ">= 132 partitions"
    img = ws.int_ws[: plan.int_ws_bytes_used].cpu().numpy().view(np.int32)
    ref_img = plan_ref.plan_image(wl.table.kv_indptr, wl.table.kv_last_page_len,
                                  page_size=64, tile_tokens=16,
                                  num_ctas=plan.problem.num_ctas, min_chunks=132,
                                  num_qo_heads=64)
    assert img.tobytes() == ref_img.tobytes()
    _, _, _, merge_indptr, _ = _decode(ref_img)
    assert min(np.diff(merge_indptr)) >= 132
    rows = _sample_rows(wl, 40, 5)
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)
    print("longctx", gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows))


def _decode(img):
    from tests.test_plan_ref import decode_image
    return decode_image(img)


def test_cascade_prefix_suffix_merge():
    wl = _workload("cascade")
    dev = gh.DeviceBatch(wl)
    pre_out, pre_lse, _, _, st1 = gh.run_pkd(dev, wl.extra_tables["prefix"])
    suf_out, suf_lse, _, _, st2 = gh.run_pkd(dev, wl.extra_tables["suffix"])
    assert st1 == 0 and st2 == 0
    out, lse = pkd.merge_states(pre_out, pre_lse, suf_out, suf_lse)
    torch.cuda.synchronize()
    rows = _sample_rows(wl, 300, 6)
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)
    print("cascade", gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows))
    # the merge alone, against the oracle merge of the GPU's own two states
    po = pre_out.float().cpu().numpy().reshape(-1, 128)[rows]
    so = suf_out.float().cpu().numpy().reshape(-1, 128)[rows]
    v_ref, s_ref = oracle.merge(po, pre_lse.cpu().numpy().reshape(-1)[rows],
                                so, suf_lse.cpu().numpy().reshape(-1)[rows])
    gh.compare(out, lse, v_ref, s_ref, wl.dtype, rows=rows)


@pytest.mark.parametrize("num_ctas,m", [(1, 1), (7, 1), (152, 1), (300, 1),
                                        (152, 9), (152, 12), (16, 40), (8, 200)])
def test_split_geometries(num_ctas, m):
    lengths = [1, 700, 0, 2049, 16, 333, 4096, 17]
    wl = workloads.make_paged("geom", lengths, num_qo_heads=32, num_kv_heads=8,
                              page_size=16, dtype="bf16", seed=7, pool_pages=700)
    dev = gh.DeviceBatch(wl)
    out, lse, plan, ws, status = gh.run_pkd(dev, num_ctas=num_ctas, min_chunks=m)
    assert status == 0
    img = ws.int_ws[: plan.int_ws_bytes_used].cpu().numpy().view(np.int32)
    ref_img = plan_ref.plan_image(wl.table.kv_indptr, wl.table.kv_last_page_len,
                                  page_size=16, tile_tokens=16, num_ctas=num_ctas,
                                  min_chunks=m, num_qo_heads=32)
    assert img.tobytes() == ref_img.tobytes()
    ref_out, ref_lse = gh.oracle_ref(wl)
    gh.compare(out, lse, ref_out, ref_lse, wl.dtype)


@pytest.mark.parametrize("hkv,hq,page", [(1, 16, 3), (2, 8, 16), (4, 32, 1), (4, 4, 64)])
def test_head_layouts(hkv, hq, page):
    lengths = [37, 0, 513, 1, 260]
    wl = workloads.make_paged("heads", lengths, num_qo_heads=hq, num_kv_heads=hkv,
                              page_size=page, dtype="f16", seed=hkv * 100 + hq)
    dev = gh.DeviceBatch(wl)
    for num_ctas, m in ((0, 1), (5, 3)):
        out, lse, plan, ws, status = gh.run_pkd(dev, num_ctas=num_ctas, min_chunks=m)
        assert status == 0
        ref_out, ref_lse = gh.oracle_ref(wl)
        gh.compare(out, lse, ref_out, ref_lse, wl.dtype)


@pytest.mark.parametrize("page,dtype", [(16, "f16"), (64, "bf16"), (32, "f16")])
def test_both_loaders_match_the_oracle(page, dtype):
    # TMA tiled boxes and per-token bulk rows on the same pages
    lengths = [5, 1000, 0, 64, 333, 2048, 16]
    used = sum((n + page - 1) // page for n in lengths)
    wl = workloads.make_paged("loaders", lengths, num_qo_heads=32, num_kv_heads=8,
                              page_size=page, dtype=dtype, seed=page, pool_pages=used + 7)
    dev = gh.DeviceBatch(wl)
    ref_out, ref_lse = gh.oracle_ref(wl)
    outs = []
    for loader in (pkd.LOADER_TMA_TILES, pkd.LOADER_BULK_ROWS):
        out, lse, _, _, status = gh.run_pkd(dev, num_ctas=40, kv_loader=loader)
        assert status == 0
        gh.compare(out, lse, ref_out, ref_lse, wl.dtype)
        outs.append((out, lse))
    # same tiles, same arithmetic: the two loaders agree bit for bit
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_tma_loader_refuses_partial_tile_pages():
    prob = pkd.make_problem(batch=1, num_qo_heads=8, num_kv_heads=8, page_size=8,
                            dtype="f16", num_pages=4, num_ctas=4,
                            kv_loader=pkd.LOADER_TMA_TILES)
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_host(prob, np.array([0, 1], np.int32), np.array([3], np.int32))
    assert e.value.status == -4


def test_plan_reuse_is_deterministic():
    wl = workloads.make_paged("reuse", [900, 33, 4000], num_qo_heads=32,
                              num_kv_heads=8, page_size=16, dtype="f16", seed=3)
    dev = gh.DeviceBatch(wl)
    out1, lse1, plan, ws, _ = gh.run_pkd(dev, num_ctas=20)
    indptr, indices, last = gh.device_table(wl.table)
    out2, lse2 = ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, wl.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_sm_scale_is_applied():
    wl = workloads.make_paged("scale", [300], num_qo_heads=8, num_kv_heads=8,
                              page_size=16, dtype="f16", seed=4)
    dev = gh.DeviceBatch(wl)
    out, lse, _, _, _ = gh.run_pkd(dev, sm_scale=0.37)
    ref_out, ref_lse = gh.oracle_ref(wl, sm_scale=0.37)
    gh.compare(out, lse, ref_out, ref_lse, wl.dtype)


def test_device_checks_flag_and_skip():
    wl = workloads.make_paged("checks", [40, 40], num_qo_heads=8, num_kv_heads=8,
                              page_size=16, dtype="f16", seed=5, pool_pages=8)
    dev = gh.DeviceBatch(wl)
    # (a) a page id out of the pool: planned without host indices, so only
    # the kernel's own range check sees it; that load is skipped
    bad = workloads.PageTable(wl.table.kv_indptr.copy(), wl.table.kv_indices.copy(),
                              wl.table.kv_last_page_len.copy(), 16)
    bad.kv_indices[1] = 1000
    prob = pkd.make_problem(batch=2, num_qo_heads=8, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=wl.num_pages)
    ws = pkd.Workspace(prob)
    plan = ws.plan(bad.kv_indptr, bad.kv_last_page_len, None)
    indptr, indices, last = gh.device_table(bad)
    ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, wl.sm_scale)
    assert pkd.check_status(ws.int_ws) & pkd.DEVICE_BAD_PAGE
    # (b) a plan made for longer requests than the device table holds: the
    # kernel clamps the units to the device lengths and flags it
    plan = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, None)
    short_last = torch.tensor([1, 1], dtype=torch.int32, device="cuda")
    indptr, indices, _ = gh.device_table(wl.table)
    ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, short_last, wl.sm_scale)
    assert pkd.check_status(ws.int_ws) & pkd.DEVICE_BAD_LENGTH
    # (c) a workspace that holds no plan image
    ws2 = pkd.Workspace(prob)
    plan2 = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, None)
    ws2.run(plan2, dev.q, dev.k, dev.v, indptr, indices,
            gh.device_table(wl.table)[2], wl.sm_scale)
    assert pkd.check_status(ws2.int_ws) & pkd.DEVICE_BAD_PLAN
    # a clean plan afterwards resets the word
    plan = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, None)
    ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, gh.device_table(wl.table)[2],
           wl.sm_scale)
    assert pkd.check_status(ws.int_ws) == 0


def test_unit_off_a_tile_boundary_is_refused():
    # a plan unit must start on a tile boundary: one planted in the device copy
    # of the image (t0 = 1) is flagged and skipped, the other requests are
    # untouched
    wl = workloads.make_paged("misaligned", [100, 500, 900, 33], num_qo_heads=32,
                              num_kv_heads=8, page_size=16, dtype="f16", seed=8)
    dev = gh.DeviceBatch(wl)
    prob = pkd.make_problem(batch=4, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=wl.num_pages, num_ctas=4)
    ws = pkd.Workspace(prob)
    plan = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, wl.table.kv_indices)
    img = ws.int_ws[: plan.int_ws_bytes_used].cpu().numpy().view(np.int32)
    num_ctas = int(img[3])
    units = 16 + num_ctas + 1
    first = [u for u in range(int(img[4])) if img[units + 4 * u] == 0][0]
    assert img[units + 4 * first + 1] == 0 and img[units + 4 * first + 3] == -1
    ws.int_ws.view(torch.int32)[units + 4 * first + 1] = 1
    indptr, indices, last = gh.device_table(wl.table)
    out, lse = ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, wl.sm_scale)
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) & pkd.DEVICE_BAD_PLAN
    rows = np.arange(wl.num_qo_heads, 4 * wl.num_qo_heads, dtype=np.int64)
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)
    gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows)


def test_run_rejects_bad_arguments():
    wl = workloads.make_paged("args", [400], num_qo_heads=8, num_kv_heads=8,
                              page_size=16, dtype="f16", seed=6)
    dev = gh.DeviceBatch(wl)
    prob = pkd.make_problem(batch=1, num_qo_heads=8, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=wl.num_pages, num_ctas=4)
    ws = pkd.Workspace(prob)
    plan = ws.plan(wl.table.kv_indptr, wl.table.kv_last_page_len, wl.table.kv_indices)
    assert plan.num_partials == 4
    indptr, indices, last = gh.device_table(wl.table)
    with pytest.raises(pkd.PkdError) as e:
        ws.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, -1.0)
    assert e.value.status == -1
    # q starting 2 bytes past a 16-byte boundary: refused before any launch
    buf = torch.empty(dev.q.numel() + 8, dtype=dev.q.dtype, device="cuda")
    q_mis = buf[1:1 + dev.q.numel()].view(dev.q.shape)
    q_mis.copy_(dev.q)
    with pytest.raises(pkd.PkdError) as e:
        ws.run(plan, q_mis, dev.k, dev.v, indptr, indices, last, wl.sm_scale)
    assert e.value.status == -4
    with pytest.raises(pkd.PkdError) as e:
        pkd.run(plan, dev.q, dev.k, dev.v, indptr, indices, last, ws.int_ws,
                ws.float_ws[:16], wl.sm_scale)
    assert e.value.status == -3


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_states_hold_every_request_in_fp32(dtype):
    """pkd_run_decode_states: split requests' partial states in their plan
    slots (folded here by the oracle's merge), every other request's state in
    slot num_partials + b; each request's fp32 state against the oracle, the
    empty request exactly (0, -inf) ("FlashInfer" (aiwiki.ai/wiki/flashinfer),
    "Attention states")."""
    from tests.test_plan_ref import decode_image
    lengths = [0, 1, 700, 33, 2500, 16, 4000, 130]
    hq = 32
    wl = workloads.make_paged("states", lengths, num_qo_heads=hq, num_kv_heads=8,
                              page_size=16, dtype=dtype, seed=11)
    dev = gh.DeviceBatch(wl)
    prob = pkd.make_problem(batch=wl.batch, num_qo_heads=hq, num_kv_heads=8, page_size=16,
                            dtype=dtype, num_pages=wl.num_pages, num_ctas=20)
    ws = pkd.Workspace(prob)
    t = wl.table
    plan = ws.plan(t.kv_indptr, t.kv_last_page_len, t.kv_indices)
    assert 0 < plan.num_split_requests < wl.batch
    ws.run(plan, dev.q, dev.k, dev.v, *gh.device_table(t), wl.sm_scale,
           phase="decode_states")
    torch.cuda.synchronize()
    assert pkd.check_status(ws.int_ws) == 0
    slot_floats = hq * 128 + (hq + 3) // 4 * 4
    nslots = plan.num_partials + wl.batch
    f = ws.float_ws[: nslots * slot_floats * 4].view(torch.float32).cpu().numpy()
    f = f.reshape(nslots, slot_floats).astype(np.float64)
    o, s = f[:, : hq * 128].reshape(nslots, hq, 128), f[:, hq * 128: hq * 128 + hq]
    _, image = pkd.plan_host(prob, t.kv_indptr, t.kv_last_page_len)
    _, _, _, merge_indptr, merge_req = decode_image(image)
    ref_out, ref_lse = gh.oracle_ref(wl)
    ref_out, ref_lse = ref_out.reshape(wl.batch, hq, 128), ref_lse.reshape(wl.batch, hq)
    for b in range(wl.batch):
        if b in merge_req:
            i = merge_req.index(b)
            slots = range(merge_indptr[i], merge_indptr[i + 1])
            v, lse = o[slots[0]], s[slots[0]]
            for j in slots[1:]:
                v, lse = oracle.merge(v, lse, o[j], s[j])
        else:
            v, lse = o[plan.num_partials + b], s[plan.num_partials + b]
        if lengths[b] == 0:
            assert np.all(v == 0.0) and np.all(lse == -np.inf), b
            continue
        assert np.abs(v - ref_out[b]).max() <= gh.OUT_TOL, b
        assert np.abs(lse - ref_lse[b]).max() <= gh.LSE_TOL, b
