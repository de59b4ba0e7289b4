"""The benchmark's own launch configuration against the oracle.

bench.py times each workload through its Runner: two workspace turns,
graph-replayed steps, and one of two copy schedules (plan images copied on a
side stream with pkd_plan, or a graph per step holding pkd_copy_plan).  The
parity tests elsewhere launch eagerly; here the Runner takes several steps,
as in the timed passes, and the result of its last step is compared with the
fp64 oracle (every row of the small workloads, sampled rows of the large
ones).
"""
import numpy as np
import pytest
import torch

import bench
from paged_kv_decode_plan_gb300 import workloads
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _check(runner, wl, rows=None):
    torch.cuda.synchronize()
    assert runner.status() == 0
    out, lse, _ = runner.result()
    ref_out, ref_lse = gh.oracle_ref(wl, rows=rows)
    return gh.compare(out, lse, ref_out, ref_lse, wl.dtype, rows=rows)


def _sample(wl, n, seed):
    rng = np.random.default_rng(seed)
    total = wl.batch * wl.num_qo_heads
    rows = set(rng.choice(total, size=min(n, total), replace=False).tolist())
    rows.update([0, total - 1])
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["single", "batch64", "cascade"])
@pytest.mark.parametrize("copies", ["side", "graph"])
def test_bench_runner_matches_oracle(name, copies):
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    wl = workloads.WORKLOADS[name]()
    runner = bench.Runner(wl, torch.device("cuda", 0), graph=True, copies=copies)
    for _ in range(7):   # eager steps, captures, replays on both turns
        runner.step()
    rows = _sample(wl, 300, 3) if name == "cascade" else None
    _check(runner, wl, rows)
    # a timed step (events inside the graph) leaves the same result
    events = tuple(torch.cuda.Event(enable_timing=True) for _ in range(4))
    runner.step(events)
    _check(runner, wl, rows)


@pytest.mark.parametrize("name,copies", [("single", "graph"), ("single", "side"),
                                         ("cascade", "side")])
def test_bench_runner_end_to_end_step_matches_oracle(name, copies):
    """A step with host inputs copied in and the result read back into pinned
    memory (the e2e loop's step): one graph per step, or the copies on their
    own streams beside the kernels' graph."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    wl = getattr(workloads, name)()
    runner = bench.Runner(wl, torch.device("cuda", 0), graph=True, copies=copies)
    in_h = runner.host_inputs()
    res_bytes = runner.result()[2].numel()
    outs = [torch.empty(res_bytes, dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    for _ in range(7):
        runner.step(inputs=in_h, outputs=outs[runner.turn])
    torch.cuda.synchronize()
    assert torch.equal(outs[runner.last_turn], runner.result()[2].cpu())
    _check(runner, wl, None if name == "single" else _sample(wl, 100, 6))


@pytest.mark.parametrize("name", ["longtail", "longctx"])
def test_bench_runner_large_workloads_sampled(name):
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    wl = workloads.WORKLOADS[name]()
    runner = bench.Runner(wl, torch.device("cuda", 0), graph=True, copies="side")
    for _ in range(5):
        runner.step()
    print(name, _check(runner, wl, _sample(wl, 48, 4)))


@pytest.mark.parametrize("layout,loader", [("hnd", 0), ("nhd", 1), ("nhd", 2), ("hnd", 2)])
def test_bench_runner_layouts_and_loaders(layout, loader):
    """batch-64 through the Runner with HND pages (the bench transposes the
    same values) and each K/V loader."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    wl = workloads.batch64()
    runner = bench.Runner(wl, torch.device("cuda", 0), graph=True, copies="side",
                          layout=layout, kv_loader=loader)
    for _ in range(6):
        runner.step()
    _check(runner, wl)


@pytest.mark.parametrize("cascade", ["shared", "per-request"])
def test_bench_runner_cascade_modes(cascade):
    """The composed cascade (prefix run + suffix run + merge_states) and the
    prefix listed in every request's table."""
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    wl = workloads.cascade()
    runner = bench.Runner(wl, torch.device("cuda", 0), graph=True, copies="side",
                          cascade=cascade)
    for _ in range(6):
        runner.step()
    _check(runner, wl, _sample(wl, 200, 5))
