"""The timeout status path of the decode kernel, with the failure made on the
host: the test hook PKD_TEST_INJECT leaves one role of every CTA out (the
loader warp, or the consumer warps); in its place one thread raises the CTA's
abort flag after about 100 us, as a warp whose wait ran out does.  The other
role's waits must then give up, record PKD_DEVICE_TIMEOUT in the status word
and retire every CTA (the loader waits for each copy it issued before its CTA
exits), so that the context stays usable: the next, normal run on the same
inputs must match the oracle.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_plan_gb300 as pkd
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def batch():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    # every CTA of an 8-CTA plan gets far more tiles than its ring has stages,
    # so a loader without consumers runs into a full ring
    wl = workloads.make_paged("timeout", [4096, 3000, 2500, 4000], num_qo_heads=32,
                              num_kv_heads=8, page_size=16, dtype="f16", seed=31)
    return wl, gh.DeviceBatch(wl)


@pytest.mark.parametrize("loader", [pkd.LOADER_TMA_TILES, pkd.LOADER_BULK_ROWS])
@pytest.mark.parametrize("mode", ["no-loader", "no-consumers"])
def test_wait_timeout_is_reported_and_context_stays_usable(batch, mode, loader, monkeypatch):
    wl, dev = batch
    monkeypatch.setenv("PKD_TEST_INJECT", mode)
    _, _, _, _, status = gh.run_pkd(dev, num_ctas=8, kv_loader=loader)
    assert status & pkd.DEVICE_TIMEOUT, status
    monkeypatch.delenv("PKD_TEST_INJECT")
    out, lse, _, _, status = gh.run_pkd(dev, num_ctas=8, kv_loader=loader)
    assert status == 0
    ref_out, ref_lse = gh.oracle_ref(wl)
    gh.compare(out, lse, ref_out, ref_lse, wl.dtype)
