"""Shared helpers for the GPU parity tests: run a batch through the C ABI,
compute the oracle on the same inputs, compare within the stated bounds.

Bounds (fp16 / bf16 inputs, fp32 accumulation):
* out: |out - ref| <= 5e-3 where |ref| < 2; where |ref| >= 2 the output type's
  own half-ulp is added (bf16 spacing there is >= 2^-6, so no bf16 value can
  be within 5e-3 of every real number), and such elements are counted apart.
* lse: |lse - ref| <= 1e-3 + 2 ulp_fp32(|ref|); the second term only matters
  beyond |lse| = 2^13, where fp32 itself cannot resolve 1e-3.
* empty rows: out exactly 0 and lse exactly -inf.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads

OUT_TOL = 5e-3
LSE_TOL = 1e-3


def device_table(table, device="cuda"):
    return (torch.from_numpy(table.kv_indptr).to(device),
            torch.from_numpy(table.kv_indices if table.kv_indices.size else
                             np.zeros(1, np.int32)).to(device),
            torch.from_numpy(table.kv_last_page_len if table.kv_last_page_len.size
                             else np.zeros(1, np.int32)).to(device))


class DeviceBatch:
    """A PagedBatch's tensors on the GPU."""

    def __init__(self, wl: workloads.PagedBatch, device="cuda"):
        self.wl = wl
        self.q = wl.q.to(device)
        self.k = wl.k_pages.to(device)
        self.v = wl.v_pages.to(device)


def run_pkd(dev: DeviceBatch, table=None, *, num_ctas=0, min_chunks=None,
            sm_scale=None, ws=None, q=None, kv_loader=0):
    wl = dev.wl
    table = wl.table if table is None else table
    prob = pkd.make_problem(
        batch=table.batch, num_qo_heads=wl.num_qo_heads, num_kv_heads=wl.num_kv_heads,
        page_size=table.page_size, dtype=wl.dtype, num_pages=wl.num_pages,
        num_ctas=num_ctas,
        min_chunks_per_request=wl.min_chunks_per_request if min_chunks is None
        else min_chunks, kv_loader=kv_loader)
    ws = ws or pkd.Workspace(prob)
    plan = ws.plan(table.kv_indptr, table.kv_last_page_len, table.kv_indices)
    indptr, indices, last = device_table(table)
    out, lse = ws.run(plan, dev.q if q is None else q, dev.k, dev.v, indptr, indices,
                      last, wl.sm_scale if sm_scale is None else sm_scale)
    torch.cuda.synchronize()
    status = pkd.check_status(ws.int_ws)
    return out, lse, plan, ws, status


def oracle_ref(wl, table=None, rows=None, sm_scale=None, q=None):
    table = wl.table if table is None else table
    q = wl.q if q is None else q
    return oracle.decode(workloads.as_codes(q), workloads.as_codes(wl.k_pages),
                         workloads.as_codes(wl.v_pages), table.kv_indptr,
                         table.kv_indices, table.kv_last_page_len, dtype=wl.dtype,
                         sm_scale=wl.sm_scale if sm_scale is None else sm_scale,
                         rows=rows)


def half_ulp(x, dtype):
    """Half the spacing of the output type at |x| (normal range)."""
    bits = 8 if dtype == "bf16" else 11     # significand bits incl. the implicit 1
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 0.5 * np.exp2(e - (bits - 1))


def log_accuracy(summary, dtype):
    """Appends a comparison's error summary, with the test that made it, to
    the JSON-lines file named by PKD_ACCURACY_LOG (if set)."""
    path = os.environ.get("PKD_ACCURACY_LOG")
    if not path:
        return
    rec = dict(summary, dtype=dtype,
               test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def compare(out, lse, ref_out, ref_lse, dtype, rows=None):
    """Checks GPU (out, lse) against the oracle; returns an error summary."""
    o = out.float().cpu().numpy().astype(np.float64)
    s = lse.float().cpu().numpy().astype(np.float64)
    d = o.shape[-1]
    o = o.reshape(-1, d)
    s = s.reshape(-1)
    if rows is not None:
        o, s = o[rows], s[rows]
    empty = ref_lse == -np.inf
    assert np.all(s[empty] == -np.inf), "empty rows must have lse = -inf"
    assert np.all(o[empty] == 0.0), "empty rows must have out = 0"
    assert np.all(np.isfinite(o)), "non-finite output"
    ne = ~empty
    summary = {"rows": int(ne.sum()), "max_err_out": 0.0, "max_err_lse": 0.0,
               "n_large": 0}
    if not ne.any():
        return summary
    ro, rs = ref_out[ne], ref_lse[ne]
    err = np.abs(o[ne] - ro)
    large = np.abs(ro) >= 2.0
    bound = OUT_TOL + np.where(large, half_ulp(ro, dtype), 0.0)
    lse_err = np.abs(s[ne] - rs)
    lse_bound = LSE_TOL + 2.0 * np.spacing(np.abs(rs).astype(np.float32)).astype(np.float64)
    summary.update(max_err_out=float(err.max()),
                   max_err_out_small=float(err[~large].max()) if (~large).any() else 0.0,
                   max_err_out_large=float(err[large].max()) if large.any() else 0.0,
                   max_err_lse=float(lse_err.max()), n_large=int(large.sum()),
                   n_elements=int(err.size))
    log_accuracy(summary, dtype)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), "out error %.3g at %s (ref %.4g)" % (
        err[worst], worst, ro[worst])
    assert np.all(lse_err <= lse_bound), "lse error %.3g" % lse_err.max()
    return summary
