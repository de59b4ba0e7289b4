"""bench.py's host-side arithmetic, checked without a GPU."""
import types

import bench
from paged_kv_decode_plan_gb300 import workloads


def _runner(wl, ctas):
    class Props:
        multi_processor_count = 152

    cuda = types.SimpleNamespace(get_device_properties=lambda device: Props())
    return types.SimpleNamespace(wl=wl, cascade_ctas=(ctas, 152 - ctas if ctas else 0),
                                 torch=types.SimpleNamespace(cuda=cuda), device=None)


def test_prefix_roofline_counts_both_contractions_of_the_shared_prefix():
    # 128 requests x 32 query heads against an 8192-token prefix, D 128:
    # Q K^T and P V, 2 flops per multiply-add each
    wl = workloads.cascade()
    r = bench.prefix_roofline(_runner(wl, 48), 0.05)
    assert r["algorithmic_flops_per_launch"] == 4 * 128 * 32 * 8192 * 128
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    achieved = 4 * 128 * 32 * 8192 * 128 / 50e-6 / 1e12
    assert abs(r["achieved"] - achieved) < 0.06
    assert abs(r["frac"] - achieved / r["peak"]) < 1e-4
    # the prefix plan gets 48 of 152 SMs beside the suffix decode
    assert abs(r["frac_of_its_sms"] - achieved / (r["peak"] * 48 / 152)) < 1e-4


def test_prefix_roofline_on_all_sms_has_no_share():
    r = bench.prefix_roofline(_runner(workloads.cascade(), 0), 0.03)
    assert "frac_of_its_sms" not in r and "ctas" not in r
