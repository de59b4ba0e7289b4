"""The C ABI used from plain C: tests/c/plan_from_c.c is compiled with gcc
against include/pkd.h and linked against libpkd.so; its plans (split-KV and
shared-prefix, host only, no GPU needed) must equal the Python binding's, and
a bad page id must come back as PKD_ERR_PAGE_TABLE."""
import os
import subprocess

import numpy as np
import pytest

import paged_kv_decode_plan_gb300 as pkd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plans_from_c_match_the_binding(tmp_path):
    pkd.load()
    exe = str(tmp_path / "plan_from_c")
    lib_dir = os.path.dirname(pkd.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "plan_from_c.c"), "-o", exe,
           "-L", lib_dir, "-l:libpkd.so", "-Wl,-rpath," + lib_dir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        pytest.fail("gcc failed:\n" + res.stderr)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = {l.split()[0]: l.split()[1:] for l in out.stdout.splitlines()}

    prob = pkd.make_problem(batch=3, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=64, num_ctas=7,
                            min_chunks_per_request=2)
    indptr = np.array([0, 5, 5, 7], np.int32)
    last = np.array([9, 1, 16], np.int32)
    indices = np.array([3, 17, 40, 2, 63, 11, 12], np.int32)
    plan, image = pkd.plan_host(prob, indptr, last, indices)
    assert [int(x) for x in lines["plan"]] == [plan.num_units, plan.num_partials,
                                               plan.num_split_requests, plan.total_tokens,
                                               plan.int_ws_bytes_used]
    assert [int(x) for x in lines["image"]] == image.tolist()
    assert int(lines["bad_page"][0]) == -2

    pprob = pkd.make_problem(batch=3, num_qo_heads=32, num_kv_heads=8, page_size=16,
                             dtype="f16", num_pages=64, num_ctas=16)
    pplan, pimage = pkd.plan_shared_prefix_host(pprob, np.array([4, 9, 2], np.int32), 5)
    assert [int(x) for x in lines["prefix"]] == [pplan.prefix_len, pplan.chunks,
                                                 pplan.chunk_tiles, pplan.row_tiles]
    assert [int(x) for x in lines["pimage"]] == pimage.tolist()
