"""Page append on the GPU: bit-exact against oracle.append_ref, then one full
decode step (append the new token of every request, decode over the extended
table) against the attention oracle."""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from oracle import append_ref
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _pool(lengths, page, dtype, seed, extra=4):
    wl = workloads.make_paged("append", lengths, num_qo_heads=32, num_kv_heads=8,
                              page_size=page, dtype=dtype, seed=seed,
                              pool_pages=sum((n + page - 1) // page for n in lengths) + extra)
    return wl


def _problem(wl, table):
    return pkd.make_problem(batch=table.batch, num_qo_heads=wl.num_qo_heads,
                            num_kv_heads=wl.num_kv_heads, page_size=table.page_size,
                            dtype=wl.dtype, num_pages=wl.num_pages)


@pytest.mark.parametrize("page,dtype", [(16, "f16"), (1, "bf16"), (64, "bf16"), (5, "f16")])
def test_append_is_bit_exact(page, dtype):
    lengths = [33, 1, 200, 64, 7]
    wl = _pool(lengths, page, dtype, seed=page)
    rng = np.random.default_rng(page)
    t = wl.table
    # every request gets tokens at random positions inside its length
    bi, pos = [], []
    for b, n in enumerate(lengths):
        for p in rng.choice(n, size=min(n, 9), replace=False):
            bi.append(b)
            pos.append(int(p))
    bi = np.array(bi, np.int32)
    pos = np.array(pos, np.int32)
    kn = workloads._fill_normal((bi.size, 8, 128), dtype, 77, 5)
    vn = workloads._fill_normal((bi.size, 8, 128), dtype, 77, 6)
    k_ref, v_ref, skipped = append_ref.append_kv(
        workloads.as_codes(wl.k_pages), workloads.as_codes(wl.v_pages),
        workloads.as_codes(kn), workloads.as_codes(vn), bi, pos, t.kv_indptr,
        t.kv_indices, t.kv_last_page_len)
    assert skipped == []
    k_dev, v_dev = wl.k_pages.cuda(), wl.v_pages.cuda()
    dev_table = gh.device_table(t)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(_problem(wl, t), kn.cuda(), vn.cuda(), torch.from_numpy(bi).cuda(),
                  torch.from_numpy(pos).cuda(), k_dev, v_dev, *dev_table, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(workloads.as_codes(k_dev.cpu()), k_ref)
    assert np.array_equal(workloads.as_codes(v_dev.cpu()), v_ref)


def test_append_skips_and_flags_out_of_range_tokens():
    wl = _pool([20, 3], 16, "f16", seed=3)
    t = wl.table
    k_dev, v_dev = wl.k_pages.cuda(), wl.v_pages.cuda()
    before = k_dev.clone()
    kn = torch.ones(3, 8, 128, dtype=torch.float16, device="cuda")
    bi = torch.tensor([0, 5, 1], dtype=torch.int32, device="cuda")   # request 5: none
    pos = torch.tensor([20, 0, 3], dtype=torch.int32, device="cuda")  # 20, 3: past end
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkd.append_kv(_problem(wl, t), kn, kn, bi, pos, k_dev, v_dev, *gh.device_table(t),
                  status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pkd.DEVICE_BAD_LENGTH
    assert torch.equal(k_dev, before)


@pytest.mark.parametrize("page,dtype", [(16, "f16"), (1, "bf16")])
def test_decode_step_after_append(page, dtype):
    # cache before the step, then one new token per request
    lengths = [16, 100, 31, 1, 257]
    wl = _pool(lengths, page, dtype, seed=11, extra=8)
    old = wl.table
    # extend each request by one token: a fresh page when its last one is full
    free = sorted(set(range(wl.num_pages)) - set(old.kv_indices.tolist()))
    new_indptr, new_indices = [0], []
    for b, n in enumerate(lengths):
        pages = list(old.kv_indices[old.kv_indptr[b]:old.kv_indptr[b + 1]])
        if n % page == 0:
            pages.append(free.pop(0))
        new_indices += pages
        new_indptr.append(len(new_indices))
    new_lengths = [n + 1 for n in lengths]
    new_last = [n - (new_indptr[b + 1] - new_indptr[b] - 1) * page
                for b, n in enumerate(new_lengths)]
    table = workloads.PageTable(np.array(new_indptr, np.int32),
                                np.array(new_indices, np.int32),
                                np.array(new_last, np.int32), page)
    bi = np.arange(len(lengths), dtype=np.int32)
    pos = np.array(lengths, np.int32)  # the new token's position
    kn = workloads._fill_normal((len(lengths), 8, 128), dtype, 91, 5)
    vn = workloads._fill_normal((len(lengths), 8, 128), dtype, 91, 6)

    dev = gh.DeviceBatch(wl)
    dev_table = gh.device_table(table)
    pkd.append_kv(_problem(wl, table), kn.cuda(), vn.cuda(), torch.from_numpy(bi).cuda(),
                  torch.from_numpy(pos).cuda(), dev.k, dev.v, *dev_table)
    out, lse, _, _, status = gh.run_pkd(dev, table, num_ctas=12)
    assert status == 0

    k_ref, v_ref, _ = append_ref.append_kv(
        workloads.as_codes(wl.k_pages), workloads.as_codes(wl.v_pages),
        workloads.as_codes(kn), workloads.as_codes(vn), bi, pos, table.kv_indptr,
        table.kv_indices, table.kv_last_page_len)
    import oracle
    ref_out, ref_lse = oracle.decode(workloads.as_codes(wl.q), k_ref, v_ref,
                                     table.kv_indptr, table.kv_indices,
                                     table.kv_last_page_len, dtype=dtype,
                                     sm_scale=wl.sm_scale)
    gh.compare(out, lse, ref_out, ref_lse, dtype)
