"""Host-side argument checks of the cascade entry points (no GPU needed).

pkd_run_cascade, pkd_run_cascade_merge, pkd_run_shared_prefix_states and
pkd_run_decode_states check plans, problem agreement, pointers and workspace sizes on the host and
return a status before any CUDA call; these tests pass placeholder device
addresses that a launch would need, so a check that let them through would
fail here loudly rather than touch memory.
"""
import ctypes

import numpy as np

import paged_kv_decode_plan_gb300 as pkd

INVALID_ARG, WORKSPACE = -1, -3
FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned placeholder, never dereferenced


def _suffix_plan(batch=3, dtype="f16"):
    prob = pkd.make_problem(batch=batch, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype=dtype, num_pages=64, num_ctas=8)
    lengths = [40, 300, 17][:batch]
    npages = [(n + 15) // 16 for n in lengths]
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.array([n - (p - 1) * 16 for n, p in zip(lengths, npages)], dtype=np.int32)
    plan, _ = pkd.plan_host(prob, indptr, last)
    return plan


def _prefix_plan(suffix, **override):
    """A prefix plan as pkd_plan_shared_prefix would describe a one-page prefix."""
    pp = pkd.PrefixPlan()
    pp.problem = pkd.Problem.from_buffer_copy(suffix.problem)
    for k, v in override.items():
        setattr(pp.problem, k, v)
    pp.prefix_len, pp.prefix_num_pages, pp.chunks, pp.chunk_tiles = 16, 1, 1, 1
    pp.row_tiles = 1
    pp.num_blocks = pp.problem.num_kv_heads
    pp.int_ws_bytes_used = 4 * 17
    pp.float_ws_bytes_needed = 4 * pp.problem.batch * (32 * 128 + 32)
    pp.valid = 1
    return pp


def _cascade(plan, pp, out=FAKE, lse=FAKE, prefix_float=FAKE, prefix_bytes=1 << 30,
             float_bytes=1 << 30):
    lib = pkd.load()
    return lib.pkd_run_cascade(ctypes.byref(plan), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                               FAKE, float_bytes, ctypes.byref(pp), FAKE, prefix_float,
                               prefix_bytes, ctypes.c_float(0.088), out, lse, None)


def _states_bytes(plan):
    """fp32 slots a states-only decode needs: the plan's partial slots plus
    one per request."""
    return (plan.num_partials + plan.problem.batch) * 4 * (32 * 128 + 32)


def _message():
    return pkd.load().pkd_last_error().decode()


def test_cascade_rejects_an_invalid_prefix_plan():
    plan = _suffix_plan()
    pp = _prefix_plan(plan)
    pp.valid = 0
    assert _cascade(plan, pp) == INVALID_ARG
    assert "prefix plan" in _message()


def test_cascade_rejects_plans_that_disagree():
    plan = _suffix_plan()
    for field, value in [("batch", 2), ("num_qo_heads", 64), ("dtype", pkd.PKD_BF16),
                         ("page_size", 32), ("num_pages", 65),
                         ("kv_layout", pkd.LAYOUT_HND)]:
        pp = _prefix_plan(plan, **{field: value})
        assert _cascade(plan, pp) == INVALID_ARG, field
        assert "differ" in _message(), field


def test_cascade_checks_pointers_and_prefix_workspace():
    plan = _suffix_plan()
    pp = _prefix_plan(plan)
    assert _cascade(plan, pp, out=None) == INVALID_ARG
    assert _cascade(plan, pp, prefix_float=None) == INVALID_ARG
    assert _cascade(plan, pp, prefix_bytes=pp.float_ws_bytes_needed - 1) == WORKSPACE
    assert "prefix float workspace" in _message()


def test_cascade_merge_checks_before_launching():
    plan = _suffix_plan()
    lib = pkd.load()
    pp = _prefix_plan(plan, batch=1)
    assert lib.pkd_run_cascade_merge(ctypes.byref(plan), FAKE, FAKE, 1 << 30,
                                     ctypes.byref(pp), FAKE, FAKE, 1 << 30, FAKE, FAKE,
                                     None) == INVALID_ARG
    pp = _prefix_plan(plan)
    assert lib.pkd_run_cascade_merge(ctypes.byref(plan), FAKE, FAKE, 1 << 30,
                                     ctypes.byref(pp), FAKE, FAKE, 8, FAKE, FAKE,
                                     None) == WORKSPACE


def test_prefix_states_check_the_plan_and_pointers():
    plan = _suffix_plan()
    lib = pkd.load()
    pp = _prefix_plan(plan)
    pp.valid = 0
    assert lib.pkd_run_shared_prefix_states(ctypes.byref(pp), FAKE, FAKE, FAKE, FAKE, FAKE,
                                            1 << 30, ctypes.c_float(0.088),
                                            None) == INVALID_ARG
    pp = _prefix_plan(plan)
    assert lib.pkd_run_shared_prefix_states(ctypes.byref(pp), None, FAKE, FAKE, FAKE, FAKE,
                                            1 << 30, ctypes.c_float(0.088),
                                            None) == INVALID_ARG
    assert lib.pkd_run_shared_prefix_states(ctypes.byref(pp), FAKE, FAKE, FAKE, FAKE, FAKE,
                                            8, ctypes.c_float(0.088), None) == WORKSPACE


def test_states_only_decode_checks_its_float_workspace():
    plan = _suffix_plan()
    lib = pkd.load()
    need = _states_bytes(plan)
    assert need > plan.float_ws_bytes_needed   # one slot per request on top

    def run(float_ws, nbytes):
        return lib.pkd_run_decode_states(ctypes.byref(plan), FAKE, FAKE, FAKE, FAKE, FAKE,
                                         FAKE, FAKE, float_ws, nbytes, ctypes.c_float(0.088),
                                         None)
    assert run(FAKE, need - 1) == WORKSPACE
    assert run(None, need) == WORKSPACE
    assert "float workspace" in _message()


def test_cascade_checks_the_suffix_states_workspace():
    plan = _suffix_plan()
    pp = _prefix_plan(plan)
    assert _cascade(plan, pp, float_bytes=_states_bytes(plan) - 1) == WORKSPACE
    assert "float workspace" in _message()
    lib = pkd.load()
    assert lib.pkd_run_cascade_merge(ctypes.byref(plan), FAKE, FAKE, _states_bytes(plan) - 1,
                                     ctypes.byref(pp), FAKE, FAKE, 1 << 30, FAKE, FAKE,
                                     None) == WORKSPACE


def test_plan_host_into_caller_buffer_and_guards():
    """plan_host / plan_shared_prefix_host write into a given host int32
    buffer (returned as is, the same image as a fresh plan) and refuse device
    or non-int32 buffers before calling the library."""
    import numpy as np
    import paged_kv_decode_plan_gb300 as pkd
    prob = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=16,
                            dtype="f16", num_pages=64, num_ctas=8)
    indptr = np.array([0, 3, 5], np.int32)
    last = np.array([16, 7], np.int32)
    buf = np.full(4096, -1, np.int32)
    plan, img = pkd.plan_host(prob, indptr, last, image=buf)
    assert img is buf
    _, fresh = pkd.plan_host(prob, indptr, last)
    n = plan.int_ws_bytes_used // 4
    assert np.array_equal(buf[:n], fresh)

    class FakeDevice:
        is_cuda = True
        dtype = "int32"
    for bad in (np.zeros(1024, np.int64), FakeDevice()):
        try:
            pkd.plan_host(prob, indptr, last, image=bad)
        except ValueError:
            pass
        else:
            raise AssertionError("accepted %r" % (bad,))
    pprob = pkd.make_problem(batch=2, num_qo_heads=32, num_kv_heads=8, page_size=16,
                             dtype="f16", num_pages=64, num_ctas=16)
    pbuf = np.zeros(64, np.int32)
    pplan, pimg = pkd.plan_shared_prefix_host(pprob, np.array([4, 9, 2], np.int32), 5,
                                              image=pbuf)
    assert pimg is pbuf and pplan.prefix_len == 37
    try:
        pkd.plan_shared_prefix_host(pprob, np.array([4, 9, 2], np.int32), 5,
                                    image=FakeDevice())
    except ValueError:
        pass
    else:
        raise AssertionError("accepted a device buffer")
