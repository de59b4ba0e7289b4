"""The library's C++ planner equals the plain-Python planning rule bit for bit,
and rejects malformed page tables and undersized buffers with status codes."""
import numpy as np
import pytest

import paged_kv_decode_plan_gb300 as pkd
from oracle import plan_ref
from paged_kv_decode_plan_gb300 import workloads
from tests.test_plan_ref import CASES, random_table


def problem_for(batch, page_size, hkv=8, hq=32, ctas=152, m=1, num_pages=1 << 20,
                dtype="f16", max_batch=0, tile=0):
    return pkd.make_problem(batch=batch, num_qo_heads=hq, num_kv_heads=hkv,
                            page_size=page_size, dtype=dtype, num_pages=num_pages,
                            num_ctas=ctas, min_chunks_per_request=m,
                            tile_tokens=tile, max_batch=max_batch)


HKV_FOR_CASE = [8, 8, 4, 8, 2, 1, 4, 8, 2]


@pytest.mark.parametrize("case,hkv", list(zip(CASES, HKV_FOR_CASE)))
def test_plan_matches_reference_rule(case, hkv):
    batch, page_size, max_len, _, ctas, m = case
    tile = 16
    rng = np.random.default_rng(hash(case) % (2 ** 32) + 1)
    for _ in range(3):
        _, indptr, last = random_table(rng, batch, page_size, max_len)
        prob = problem_for(batch, page_size, hkv=hkv, hq=4 * hkv, ctas=ctas, m=m)
        plan, image = pkd.plan_host(prob, indptr, last)
        ref = plan_ref.plan_image(indptr, last, page_size=page_size, tile_tokens=tile,
                                  num_ctas=ctas, min_chunks=m, num_qo_heads=4 * hkv)
        assert image.dtype == ref.dtype == np.int32
        assert image.tobytes() == ref.tobytes()
        assert plan.num_units == ref[4] and plan.num_partials == ref[5]
        assert plan.num_split_requests == ref[6] and plan.total_tiles == ref[9]
        assert plan.problem.tile_tokens == tile
        assert plan.total_tokens == int(np.sum(
            plan_ref.request_lengths(indptr, last, page_size)))
        assert plan.int_ws_bytes_used == 4 * ref.size


@pytest.mark.parametrize("name", ["single", "batch64", "longtail", "cascade", "longctx"])
def test_workload_plans_match(name):
    # page tables of the five measured workloads (no tensors generated)
    if name == "longtail":
        table = workloads.table_from_lengths(workloads.longtail_lengths(1003), 1,
                                             np.arange(1 << 24))
        hq, m = 32, 1
    elif name == "longctx":
        table = workloads.table_from_lengths([131072] * 8, 64, np.arange(1 << 16))
        hq, m = 64, 132
    elif name == "batch64":
        lengths = np.random.default_rng([1002, 0]).integers(128, 4096, 64, endpoint=True)
        table = workloads.table_from_lengths(lengths, 16, np.arange(1 << 16))
        hq, m = 32, 1
    elif name == "cascade":
        lengths = 8192 + np.random.default_rng([1004, 0]).integers(64, 1024, 128,
                                                                   endpoint=True)
        table = workloads.table_from_lengths(lengths, 16, np.arange(1 << 17))
        hq, m = 32, 1
    else:
        table = workloads.table_from_lengths([512], 16, np.arange(64))
        hq, m = 32, 1
    prob = problem_for(table.batch, table.page_size, hq=hq, m=m)
    _, image = pkd.plan_host(prob, table.kv_indptr, table.kv_last_page_len)
    ref = plan_ref.plan_image(table.kv_indptr, table.kv_last_page_len,
                              page_size=table.page_size, tile_tokens=16, num_ctas=152,
                              min_chunks=m, num_qo_heads=hq)
    assert image.tobytes() == ref.tobytes()


def expect_status(status, fn, *args, **kwargs):
    with pytest.raises(pkd.PkdError) as info:
        fn(*args, **kwargs)
    assert info.value.status == status, str(info.value)


def test_malformed_tables_are_rejected():
    prob = problem_for(2, 16, num_pages=10)
    ok_indptr = np.array([0, 2, 3], np.int32)
    ok_last = np.array([5, 16], np.int32)
    pkd.plan_host(prob, ok_indptr, ok_last, np.array([0, 1, 9], np.int32))
    expect_status(-2, pkd.plan_host, prob, np.array([0, 2, 1], np.int32), ok_last)
    expect_status(-2, pkd.plan_host, prob, np.array([-1, 2, 3], np.int32), ok_last)
    expect_status(-2, pkd.plan_host, prob, ok_indptr, np.array([0, 16], np.int32))
    expect_status(-2, pkd.plan_host, prob, ok_indptr, np.array([5, 17], np.int32))
    expect_status(-2, pkd.plan_host, prob, ok_indptr, ok_last,
                  np.array([0, 1, 10], np.int32))
    expect_status(-2, pkd.plan_host, prob, ok_indptr, ok_last,
                  np.array([0, -3, 2], np.int32))
    # an empty request ignores its last_page_len
    pkd.plan_host(prob, np.array([0, 0, 1], np.int32), np.array([0, 3], np.int32))


def test_unsupported_and_invalid_problems():
    indptr = np.array([0, 1], np.int32)
    last = np.array([3], np.int32)
    expect_status(-4, pkd.plan_host, problem_for(1, 16, hkv=3, hq=6), indptr, last)
    expect_status(-4, pkd.plan_host, problem_for(1, 16, hkv=1, hq=32), indptr, last)
    expect_status(-4, pkd.plan_host, problem_for(1, 16, dtype="f32"), indptr, last)
    expect_status(-4, pkd.plan_host, problem_for(1, 16, tile=32), indptr, last)
    expect_status(-4, pkd.plan_host, problem_for(1, 16, hkv=4, hq=8, tile=32), indptr, last)
    expect_status(-1, pkd.plan_host, problem_for(1, 16, hkv=8, hq=12), indptr, last)
    expect_status(-1, pkd.plan_host, problem_for(2, 16, max_batch=1),
                  np.array([0, 1, 2], np.int32), np.array([3, 3], np.int32))
    bad = problem_for(1, 16)
    bad.head_dim = 64
    expect_status(-4, pkd.plan_host, bad, indptr, last)


def test_capacity_bound_holds_for_extreme_splits():
    # every request minimally long for the cap-chunk count to peak
    for m in (1, 2, 7, 132):
        lengths = [16 * (2 * m - 1)] * 5 + [0, 16]
        table = workloads.table_from_lengths(lengths, 16, np.arange(10 ** 5))
        prob = problem_for(len(lengths), 16, m=m, ctas=13)
        plan, image = pkd.plan_host(prob, table.kv_indptr, table.kv_last_page_len)
        ib, fb, sb = pkd.workspace_size(prob)
        assert plan.int_ws_bytes_used <= ib and sb == ib
        assert plan.float_ws_bytes_needed <= fb
        # a states-only decode also keeps one fp32 state per unsplit request
        slot = 4 * (32 * 128 + 32)
        assert (plan.num_partials + len(lengths)) * slot <= fb
