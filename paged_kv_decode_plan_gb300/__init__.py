"""Paged KV decode attention with split-KV partial states and LSE merge (GB300).

Thin ctypes binding over the C ABI in ``include/pkd.h`` (``libpkd.so``, built
in-tree by :mod:`paged_kv_decode_plan_gb300.build`).  The functions here only
marshal arguments: every step of the computation runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  If the library is
missing, every call raises; there is no other implementation to fall back to.

Entry points (same names as the C ABI without the ``pkd_`` prefix):
``workspace_size``, ``plan_host``, ``plan``, ``copy_plan``, ``run`` (its ``phase`` picks
``pkd_run``, ``pkd_run_decode``, ``pkd_run_merge`` or
``pkd_run_decode_states``), ``run_static``, ``merge_states``,
``check_status``, the shared-prefix calls (``plan_shared_prefix``,
``plan_shared_prefix_host``, ``run_shared_prefix``, ``run_shared_prefix_states``,
``run_cascade``,
``run_cascade_merge``), ``append_kv``, plus :class:`Workspace` and
:class:`PrefixWorkspace`, which allocate the buffers a capacity needs.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkd.so")

PKD_F16, PKD_BF16, PKD_F32 = 0, 1, 2
LOADER_AUTO, LOADER_TMA_TILES, LOADER_BULK_ROWS = 0, 1, 2
LAYOUT_NHD, LAYOUT_HND = 0, 1
DEVICE_BAD_PAGE, DEVICE_BAD_LENGTH, DEVICE_BAD_PLAN, DEVICE_TIMEOUT = 1, 2, 4, 8
STATUS_NAMES = {0: "PKD_OK", -1: "PKD_ERR_INVALID_ARG", -2: "PKD_ERR_PAGE_TABLE",
                -3: "PKD_ERR_WORKSPACE", -4: "PKD_ERR_UNSUPPORTED",
                -5: "PKD_ERR_CUDA", -6: "PKD_ERR_DEVICE_CHECK"}

ABI_VERSION = 5  # PKD_ABI_VERSION of include/pkd.h

# every symbol include/pkd.h declares
EXPORTED = ("pkd_abi_version", "pkd_last_error", "pkd_workspace_size",
            "pkd_plan_host", "pkd_plan", "pkd_run", "pkd_run_decode",
            "pkd_run_merge", "pkd_merge_states", "pkd_check_status",
            "pkd_run_static", "pkd_prefix_workspace_size", "pkd_plan_shared_prefix",
            "pkd_run_shared_prefix", "pkd_append_kv", "pkd_run_shared_prefix_states",
            "pkd_run_cascade", "pkd_run_cascade_merge", "pkd_run_decode_states",
            "pkd_plan_shared_prefix_host", "pkd_copy_plan")


class PkdError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class Problem(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("num_ctas", ctypes.c_int32),
                ("min_chunks_per_request", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("kv_loader", ctypes.c_int32), ("kv_layout", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("problem", Problem), ("num_units", ctypes.c_int32),
                ("num_partials", ctypes.c_int32),
                ("num_split_requests", ctypes.c_int32),
                ("total_tiles", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("int_ws_bytes_used", ctypes.c_int64),
                ("float_ws_bytes_needed", ctypes.c_int64),
                ("valid", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class PrefixPlan(ctypes.Structure):
    _fields_ = [("problem", Problem), ("prefix_len", ctypes.c_int32),
                ("prefix_num_pages", ctypes.c_int32), ("chunks", ctypes.c_int32),
                ("chunk_tiles", ctypes.c_int32), ("row_tiles", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("int_ws_bytes_used", ctypes.c_int64),
                ("float_ws_bytes_needed", ctypes.c_int64), ("valid", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib = None


def load():
    """Loads libpkd.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libpkd.so is not built: run `python -m paged_kv_decode_plan_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    # host int32 arrays are passed as plain addresses (numpy's .ctypes view
    # costs microseconds per array, more than the planner itself)
    vp = i32p = ctypes.c_void_p
    sz = ctypes.POINTER(ctypes.c_size_t)
    lib.pkd_abi_version.restype = ctypes.c_int32
    lib.pkd_last_error.restype = ctypes.c_char_p
    lib.pkd_workspace_size.argtypes = [ctypes.POINTER(Problem), sz, sz, sz]
    lib.pkd_plan_host.argtypes = [ctypes.POINTER(Problem), i32p, i32p, i32p,
                                  ctypes.POINTER(Plan), i32p, ctypes.c_size_t]
    lib.pkd_plan.argtypes = [ctypes.POINTER(Problem), i32p, i32p, i32p,
                             ctypes.POINTER(Plan), vp, ctypes.c_size_t, vp,
                             ctypes.c_size_t, vp]
    lib.pkd_run.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, vp, vp, vp,
                            ctypes.c_size_t, ctypes.c_float, vp, vp, vp]
    lib.pkd_run_decode.argtypes = lib.pkd_run.argtypes
    lib.pkd_run_decode_states.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, vp, vp,
                                          vp, ctypes.c_size_t, ctypes.c_float, vp]
    lib.pkd_run_merge.argtypes = [ctypes.POINTER(Plan), vp, vp, ctypes.c_size_t,
                                  vp, vp, vp]
    lib.pkd_merge_states.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, vp]
    lib.pkd_check_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
    lib.pkd_run_static.argtypes = [ctypes.POINTER(Plan), i32p, vp, vp, vp, vp, vp,
                                   vp, ctypes.c_float, vp, vp, vp]
    lib.pkd_append_kv.argtypes = [ctypes.POINTER(Problem), vp, vp, vp, vp,
                                  ctypes.c_int64, vp, vp, vp, vp, vp, vp, vp]
    lib.pkd_prefix_workspace_size.argtypes = [ctypes.POINTER(Problem), ctypes.c_int32,
                                              sz, sz, sz]
    lib.pkd_plan_shared_prefix.argtypes = [ctypes.POINTER(Problem), i32p, ctypes.c_int32,
                                           ctypes.c_int32, ctypes.POINTER(PrefixPlan),
                                           vp, ctypes.c_size_t, vp, ctypes.c_size_t, vp]
    lib.pkd_plan_shared_prefix_host.argtypes = [ctypes.POINTER(Problem), i32p,
                                                ctypes.c_int32, ctypes.c_int32,
                                                ctypes.POINTER(PrefixPlan), i32p,
                                                ctypes.c_size_t]
    lib.pkd_copy_plan.argtypes = [i32p, ctypes.c_size_t, vp, ctypes.c_size_t, vp]
    lib.pkd_run_shared_prefix.argtypes = [ctypes.POINTER(PrefixPlan), vp, vp, vp, vp, vp,
                                          ctypes.c_size_t, ctypes.c_float, vp, vp, vp]
    lib.pkd_run_shared_prefix_states.argtypes = [ctypes.POINTER(PrefixPlan), vp, vp, vp,
                                                 vp, vp, ctypes.c_size_t, ctypes.c_float,
                                                 vp]
    lib.pkd_run_cascade.argtypes = [ctypes.POINTER(Plan), vp, vp, vp, vp, vp, vp, vp, vp,
                                    ctypes.c_size_t, ctypes.POINTER(PrefixPlan), vp, vp,
                                    ctypes.c_size_t, ctypes.c_float, vp, vp, vp]
    lib.pkd_run_cascade_merge.argtypes = [ctypes.POINTER(Plan), vp, vp, ctypes.c_size_t,
                                          ctypes.POINTER(PrefixPlan), vp, vp,
                                          ctypes.c_size_t, vp, vp, vp]
    for name in EXPORTED[2:]:
        getattr(lib, name).restype = ctypes.c_int
    if lib.pkd_abi_version() != ABI_VERSION:
        raise RuntimeError("libpkd.so ABI version mismatch")
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise PkdError(status, load().pkd_last_error().decode())


def abi_version() -> int:
    return int(load().pkd_abi_version())


def _dtype_code(dtype) -> int:
    import torch
    table = {torch.float16: PKD_F16, torch.bfloat16: PKD_BF16, torch.float32: PKD_F32,
             "f16": PKD_F16, "bf16": PKD_BF16, "f32": PKD_F32}
    if dtype not in table:
        raise ValueError("unsupported dtype %r" % (dtype,))
    return table[dtype]


def make_problem(*, batch, num_qo_heads, num_kv_heads, page_size, dtype,
                 num_pages, head_dim=128, num_ctas=0, min_chunks_per_request=1,
                 tile_tokens=0, max_batch=0, kv_loader=LOADER_AUTO,
                 kv_layout=LAYOUT_NHD) -> Problem:
    return Problem(batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                   _dtype_code(dtype), num_pages, num_ctas,
                   min_chunks_per_request, tile_tokens, max_batch, kv_loader,
                   {"NHD": LAYOUT_NHD, "HND": LAYOUT_HND}.get(kv_layout, kv_layout))


def workspace_size(problem: Problem):
    """(int_ws_bytes, float_ws_bytes, staging_bytes) for the problem's capacity."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().pkd_workspace_size(ctypes.byref(problem), ctypes.byref(a),
                                     ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def _host_i32(x):
    if x is None:
        return None, None
    if hasattr(x, "numpy"):
        x = x.cpu().numpy()
    a = np.ascontiguousarray(x, dtype=np.int32)
    if a.size == 0:
        a = np.zeros(1, dtype=np.int32)
    return a, _addr(a)


def _addr(a):
    """Address of a numpy array's first element (the caller keeps ``a`` alive);
    the buffer protocol is several times cheaper than numpy's ctypes view."""
    if a.flags.writeable:
        return ctypes.addressof(ctypes.c_char.from_buffer(a))
    return a.ctypes.data


def _require_host(image):
    """A host planner writes the image through a CPU pointer: refuse device
    tensors and anything that is not int32."""
    if getattr(image, "is_cuda", False):
        raise ValueError("the plan image buffer must be host memory")
    dt = getattr(image, "dtype", None)
    if dt is not None and str(dt) not in ("torch.int32", "int32"):
        raise ValueError("the plan image buffer must be int32")


def plan_host(problem: Problem, kv_indptr, kv_last_page_len, kv_indices=None, *,
              image=None):
    """Host-only planning; returns (Plan, plan image as an int32 array).

    With ``image`` (a host int32 torch tensor, e.g. pinned staging memory,
    or numpy array) the image is written into it and ``(Plan, image)`` is
    returned without a copy; otherwise a new array of the image's size.
    """
    if image is not None:
        if problem.num_ctas <= 0:
            raise ValueError("plan_host needs an explicit num_ctas")
        _require_host(image)
        if hasattr(image, "data_ptr"):
            addr, nbytes = image.data_ptr(), image.numel() * image.element_size()
        else:
            addr, nbytes = _addr(image), image.nbytes
        indptr, p_indptr = _host_i32(kv_indptr)
        last, p_last = _host_i32(kv_last_page_len)
        idx, p_idx = _host_i32(kv_indices)
        out = Plan()
        _check(load().pkd_plan_host(ctypes.byref(problem), p_indptr, p_last, p_idx,
                                    ctypes.byref(out), addr, nbytes))
        return out, image
    prob = Problem.from_buffer_copy(problem)
    if prob.num_ctas <= 0:
        raise ValueError("plan_host needs an explicit num_ctas")
    ib, _, _ = workspace_size(prob)
    image = np.zeros(ib // 4 + 1, dtype=np.int32)
    indptr, p_indptr = _host_i32(kv_indptr)
    last, p_last = _host_i32(kv_last_page_len)
    idx, p_idx = _host_i32(kv_indices)
    out = Plan()
    _check(load().pkd_plan_host(ctypes.byref(prob), p_indptr, p_last, p_idx,
                                ctypes.byref(out),
                                _addr(image),
                                image.nbytes))
    return out, image[: out.int_ws_bytes_used // 4].copy()


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t):
    # every entry point declares its pointer arguments c_void_p, so a plain
    # int is passed as a full-width address
    return None if t is None else t.data_ptr()


def plan(problem: Problem, kv_indptr, kv_last_page_len, kv_indices=None, *,
         staging, int_ws, stream=None) -> Plan:
    """Plans on the host and copies the image into ``int_ws`` on ``stream``.

    ``staging`` is a pinned host tensor of at least the staging size; it must
    not be reused before the copy has run on the stream.
    """
    indptr, p_indptr = _host_i32(kv_indptr)
    last, p_last = _host_i32(kv_last_page_len)
    idx, p_idx = _host_i32(kv_indices)
    out = Plan()
    _check(load().pkd_plan(ctypes.byref(problem), p_indptr, p_last, p_idx,
                           ctypes.byref(out), _ptr(staging),
                           staging.numel() * staging.element_size(), _ptr(int_ws),
                           int_ws.numel() * int_ws.element_size(), _stream_ptr(stream)))
    return out


def copy_plan(image, int_ws, stream=None):
    """pkd_copy_plan: a plan image in pinned host memory (an int32 torch
    tensor, e.g. a Workspace's staging buffer) into the device workspace
    ``int_ws``, by a kernel that reads the host buffer; graph-capturable."""
    _require_host(image)
    _check(load().pkd_copy_plan(_ptr(image), image.numel() * image.element_size(),
                                _ptr(int_ws), int_ws.numel() * int_ws.element_size(),
                                _stream_ptr(stream)))


def run(plan_: Plan, q, k_pages, v_pages, kv_indptr, kv_indices, kv_last_page_len,
        int_ws, float_ws, sm_scale: float, out=None, lse=None, stream=None,
        phase: str = "both"):
    """Decode attention for a planned batch; returns (out, lse).

    ``phase`` selects the C entry point: "both" (pkd_run), "decode"
    (pkd_run_decode), "merge" (pkd_run_merge; out and lse must be given) or
    "decode_states" (pkd_run_decode_states: every request's state stays fp32
    in ``float_ws``; returns None).
    """
    import torch
    p = plan_.problem
    if phase == "decode_states":
        for t in (q, k_pages, v_pages):
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
        if _dtype_code(q.dtype) != p.dtype or k_pages.dtype != q.dtype or \
                v_pages.dtype != q.dtype:
            raise ValueError("dtype does not match the plan")
        _check(load().pkd_run_decode_states(
            ctypes.byref(plan_), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indptr),
            _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(int_ws), _ptr(float_ws),
            float_ws.numel() * float_ws.element_size(), float(sm_scale),
            _stream_ptr(stream)))
        return None
    if out is None:
        out = torch.empty((p.batch, p.num_qo_heads, p.head_dim), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_qo_heads), dtype=torch.float32,
                          device=q.device)
    for t in (q, k_pages, v_pages, out):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if _dtype_code(q.dtype) != p.dtype or k_pages.dtype != q.dtype or \
            v_pages.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("dtype does not match the plan")
    if lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    fbytes = 0 if float_ws is None else float_ws.numel() * float_ws.element_size()
    lib = load()
    if phase == "merge":
        _check(lib.pkd_run_merge(ctypes.byref(plan_), _ptr(int_ws), _ptr(float_ws),
                                 fbytes, _ptr(out), _ptr(lse), _stream_ptr(stream)))
        return out, lse
    fn = {"both": lib.pkd_run, "decode": lib.pkd_run_decode}[phase]
    _check(fn(ctypes.byref(plan_), _ptr(q), _ptr(k_pages), _ptr(v_pages),
              _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len),
              _ptr(int_ws), _ptr(float_ws), fbytes, float(sm_scale),
              _ptr(out), _ptr(lse), _stream_ptr(stream)))
    return out, lse


def run_static(plan_: Plan, host_image, q, k_pages, v_pages, kv_indptr, kv_indices,
               kv_last_page_len, sm_scale: float, out=None, lse=None, stream=None):
    """pkd_run_static: decode with the library's fixed device scratch array
    instead of caller workspaces (for callers that cannot allocate device
    memory).  ``plan_`` and ``host_image`` come from :func:`plan_host`."""
    import torch
    p = plan_.problem
    if out is None:
        out = torch.empty((p.batch, p.num_qo_heads, p.head_dim), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_qo_heads), dtype=torch.float32,
                          device=q.device)
    image = np.ascontiguousarray(host_image, dtype=np.int32)
    if image.nbytes < plan_.int_ws_bytes_used:
        raise ValueError("host_image holds %d bytes; the plan image has %d"
                         % (image.nbytes, plan_.int_ws_bytes_used))
    _check(load().pkd_run_static(
        ctypes.byref(plan_), _addr(image),
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indptr), _ptr(kv_indices),
        _ptr(kv_last_page_len), float(sm_scale), _ptr(out), _ptr(lse),
        _stream_ptr(stream)))
    return out, lse


def merge_states(v_a, s_a, v_b, s_b, v_out=None, s_out=None, stream=None):
    """Merges two attention states; v: [n, H, D] (f16/bf16/f32), s: [n, H] f32."""
    import torch
    if v_a.shape != v_b.shape or s_a.shape != s_b.shape or v_a.dim() != 3 \
            or tuple(s_a.shape) != tuple(v_a.shape[:2]):
        raise ValueError("state shapes")
    if v_out is None:
        v_out = torch.empty_like(v_a)
    if s_out is None:
        s_out = torch.empty_like(s_a)
    for t in (v_a, v_b, v_out, s_a, s_b, s_out):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if v_b.dtype != v_a.dtype or v_out.dtype != v_a.dtype or s_a.dtype != torch.float32 \
            or s_b.dtype != torch.float32 or s_out.dtype != torch.float32:
        raise ValueError("dtypes")
    n, h, d = v_a.shape
    _check(load().pkd_merge_states(_ptr(v_a), _ptr(s_a), _ptr(v_b), _ptr(s_b),
                                   _ptr(v_out), _ptr(s_out), n, h, d,
                                   _dtype_code(v_a.dtype), _stream_ptr(stream)))
    return v_out, s_out


def check_status(int_ws, stream=None) -> int:
    """Device status word of a workspace (PKD_DEVICE_* bits); syncs the stream."""
    word = ctypes.c_uint32()
    st = load().pkd_check_status(_ptr(int_ws), ctypes.byref(word), _stream_ptr(stream))
    if st not in (0, -6):
        _check(st)
    return int(word.value)


def append_kv(problem: Problem, k_new, v_new, batch_indices, positions, k_pages,
              v_pages, kv_indptr, kv_indices, kv_last_page_len, status=None,
              stream=None):
    """Writes new tokens' K/V rows ([n, Hkv, D]) into the paged cache."""
    for t in (k_new, v_new, k_pages, v_pages):
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
    if k_new.dtype != k_pages.dtype or v_new.dtype != v_pages.dtype or \
            _dtype_code(k_pages.dtype) != problem.dtype:
        raise ValueError("dtype does not match the problem")
    _check(load().pkd_append_kv(
        ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(batch_indices),
        _ptr(positions), int(k_new.shape[0]), _ptr(k_pages), _ptr(v_pages),
        _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(status),
        _stream_ptr(stream)))


def prefix_workspace_size(problem: Problem, max_prefix_pages: int):
    """(int_ws_bytes, float_ws_bytes, staging_bytes) for shared prefixes."""
    a, b, c = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().pkd_prefix_workspace_size(ctypes.byref(problem), int(max_prefix_pages),
                                            ctypes.byref(a), ctypes.byref(b),
                                            ctypes.byref(c)))
    return a.value, b.value, c.value


def plan_shared_prefix_host(problem: Problem, prefix_pages, prefix_last_page_len, *,
                            image=None):
    """Host-only prefix planning; returns (PrefixPlan, image as an int32 array),
    or ``(PrefixPlan, image)`` written into the given host buffer."""
    if problem.num_ctas <= 0:
        raise ValueError("plan_shared_prefix_host needs an explicit num_ctas")
    pages, p_pages = _host_i32(prefix_pages)
    n = 0 if prefix_pages is None else int(np.asarray(prefix_pages).size)
    given = image is not None
    if given:
        _require_host(image)
    else:
        image = np.zeros(16 + n + 1, dtype=np.int32)
    if hasattr(image, "data_ptr"):
        addr, nbytes = image.data_ptr(), image.numel() * image.element_size()
    else:
        addr, nbytes = _addr(image), image.nbytes
    out = PrefixPlan()
    _check(load().pkd_plan_shared_prefix_host(
        ctypes.byref(problem), p_pages, n, int(prefix_last_page_len), ctypes.byref(out),
        addr, nbytes))
    if given:
        return out, image
    return out, image[: out.int_ws_bytes_used // 4].copy()


def plan_shared_prefix(problem: Problem, prefix_pages, prefix_last_page_len, *,
                       staging, int_ws, stream=None) -> PrefixPlan:
    """Plans attention of ``problem.batch`` requests against one shared prefix."""
    pages, p_pages = _host_i32(prefix_pages)
    n = 0 if prefix_pages is None else int(np.asarray(prefix_pages).size)
    out = PrefixPlan()
    _check(load().pkd_plan_shared_prefix(
        ctypes.byref(problem), p_pages, n, int(prefix_last_page_len), ctypes.byref(out),
        _ptr(staging), staging.numel() * staging.element_size(), _ptr(int_ws),
        int_ws.numel() * int_ws.element_size(), _stream_ptr(stream)))
    return out


def run_shared_prefix(plan_: PrefixPlan, q, k_pages, v_pages, int_ws, float_ws,
                      sm_scale: float, out=None, lse=None, stream=None):
    """States of every (request, query head) over the shared prefix."""
    import torch
    p = plan_.problem
    if out is None:
        out = torch.empty((p.batch, p.num_qo_heads, p.head_dim), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_qo_heads), dtype=torch.float32,
                          device=q.device)
    if _dtype_code(q.dtype) != p.dtype or k_pages.dtype != q.dtype or \
            v_pages.dtype != q.dtype or out.dtype != q.dtype:
        raise ValueError("dtype does not match the plan")
    _check(load().pkd_run_shared_prefix(
        ctypes.byref(plan_), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(int_ws),
        _ptr(float_ws), float_ws.numel() * float_ws.element_size(), float(sm_scale),
        _ptr(out), _ptr(lse), _stream_ptr(stream)))
    return out, lse


def run_shared_prefix_states(plan_: PrefixPlan, q, k_pages, v_pages, int_ws, float_ws,
                             sm_scale: float, stream=None):
    """The shared-prefix kernel alone: chunk states into ``float_ws``."""
    p = plan_.problem
    if _dtype_code(q.dtype) != p.dtype or k_pages.dtype != q.dtype or \
            v_pages.dtype != q.dtype:
        raise ValueError("dtype does not match the plan")
    _check(load().pkd_run_shared_prefix_states(
        ctypes.byref(plan_), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(int_ws),
        _ptr(float_ws), float_ws.numel() * float_ws.element_size(), float(sm_scale),
        _stream_ptr(stream)))


def _state_buffers(p, q, out, lse):
    import torch
    if out is None:
        out = torch.empty((p.batch, p.num_qo_heads, p.head_dim), dtype=q.dtype,
                          device=q.device)
    if lse is None:
        lse = torch.empty((p.batch, p.num_qo_heads), dtype=torch.float32,
                          device=q.device)
    if out.dtype != q.dtype or lse.dtype != torch.float32:
        raise ValueError("out must have the query dtype and lse float32")
    if not out.is_contiguous() or not lse.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return out, lse


def run_cascade(plan_: Plan, prefix_plan: PrefixPlan, q, k_pages, v_pages, kv_indptr,
                kv_indices, kv_last_page_len, ws, prefix_ws, sm_scale: float, out=None,
                lse=None, stream=None):
    """Attention over a shared prefix followed by each request's suffix.

    ``plan_`` / ``ws`` (a :class:`Workspace`) are the suffix plan and its
    buffers, ``kv_*`` the suffix pages; ``prefix_plan`` / ``prefix_ws`` (a
    :class:`PrefixWorkspace`) the shared prefix.  Returns (out, lse).
    """
    out, lse = _state_buffers(plan_.problem, q, out, lse)
    if _dtype_code(q.dtype) != plan_.problem.dtype or k_pages.dtype != q.dtype or \
            v_pages.dtype != q.dtype:
        raise ValueError("dtype does not match the plan")
    fbytes = ws.float_ws.numel() * ws.float_ws.element_size()
    pbytes = prefix_ws.float_ws.numel() * prefix_ws.float_ws.element_size()
    _check(load().pkd_run_cascade(
        ctypes.byref(plan_), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(kv_indptr),
        _ptr(kv_indices), _ptr(kv_last_page_len), _ptr(ws.int_ws), _ptr(ws.float_ws),
        fbytes, ctypes.byref(prefix_plan), _ptr(prefix_ws.int_ws),
        _ptr(prefix_ws.float_ws), pbytes, float(sm_scale), _ptr(out), _ptr(lse),
        _stream_ptr(stream)))
    return out, lse


def run_cascade_merge(plan_: Plan, prefix_plan: PrefixPlan, ws, prefix_ws, out, lse,
                      stream=None):
    """The last launch of :func:`run_cascade`: folds the prefix chunk states
    and the fp32 suffix states that ``ws.run(..., phase="decode_states")``
    left in ``ws`` into (out, lse)."""
    fbytes = ws.float_ws.numel() * ws.float_ws.element_size()
    pbytes = prefix_ws.float_ws.numel() * prefix_ws.float_ws.element_size()
    _check(load().pkd_run_cascade_merge(
        ctypes.byref(plan_), _ptr(ws.int_ws), _ptr(ws.float_ws), fbytes,
        ctypes.byref(prefix_plan), _ptr(prefix_ws.int_ws), _ptr(prefix_ws.float_ws),
        pbytes, _ptr(out), _ptr(lse), _stream_ptr(stream)))
    return out, lse


class PrefixWorkspace:
    """Workspaces and pinned staging for shared prefixes of a capacity."""

    def __init__(self, problem: Problem, max_prefix_pages: int, device=None):
        import torch
        self.problem = Problem.from_buffer_copy(problem)
        ib, fb, sb = prefix_workspace_size(self.problem, max_prefix_pages)
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.int_ws = torch.zeros(ib, dtype=torch.uint8, device=device)
        self.float_ws = torch.empty(max(fb, 16), dtype=torch.uint8, device=device)
        self.staging = torch.empty(sb // 4 + 4, dtype=torch.int32, pin_memory=True)
        self.event = torch.cuda.Event()   # re-recorded after every image copy
        self.recorded = False

    def plan(self, prefix_pages, prefix_last_page_len, *, batch=None, stream=None):
        import torch
        prob = self.problem
        if batch is not None:
            prob = Problem.from_buffer_copy(self.problem)
            prob.batch = batch
        if self.recorded:
            self.event.synchronize()
        out = plan_shared_prefix(prob, prefix_pages, prefix_last_page_len,
                                 staging=self.staging, int_ws=self.int_ws, stream=stream)
        self.event.record(stream or torch.cuda.current_stream())
        self.recorded = True
        return out

    def run(self, plan_: PrefixPlan, q, k_pages, v_pages, sm_scale, out=None, lse=None,
            stream=None):
        return run_shared_prefix(plan_, q, k_pages, v_pages, self.int_ws, self.float_ws,
                                 sm_scale, out=out, lse=lse, stream=stream)

    def run_states(self, plan_: PrefixPlan, q, k_pages, v_pages, sm_scale, stream=None):
        run_shared_prefix_states(plan_, q, k_pages, v_pages, self.int_ws, self.float_ws,
                                 sm_scale, stream=stream)


class Workspace:
    """Device workspaces and two pinned staging buffers for one capacity.

    Plans alternate between the staging buffers; before reusing one, the
    event recorded after its copy is waited on, so the host never overwrites
    an image the stream has not copied yet.
    """

    def __init__(self, problem: Problem, device=None):
        import torch
        self.problem = Problem.from_buffer_copy(problem)
        ib, fb, sb = workspace_size(self.problem)
        device = device or torch.device("cuda", torch.cuda.current_device())
        self.int_ws = torch.zeros(ib, dtype=torch.uint8, device=device)
        self.float_ws = torch.empty(max(fb, 16), dtype=torch.uint8, device=device)
        self.staging = [torch.empty(sb // 4 + 4, dtype=torch.int32, pin_memory=True)
                        for _ in range(2)]
        # one event per staging buffer, re-recorded after each of its copies
        self.events = [torch.cuda.Event(), torch.cuda.Event()]
        self.recorded = [False, False]
        self.turn = 0

    def plan(self, kv_indptr, kv_last_page_len, kv_indices=None, *, batch=None,
             stream=None) -> Plan:
        import torch
        prob = self.problem
        if batch is not None:
            prob = Problem.from_buffer_copy(self.problem)
            prob.batch = batch
        i = self.turn
        if self.recorded[i]:
            self.events[i].synchronize()
        out = plan(prob, kv_indptr, kv_last_page_len, kv_indices,
                   staging=self.staging[i], int_ws=self.int_ws, stream=stream)
        self.events[i].record(stream or torch.cuda.current_stream())
        self.recorded[i] = True
        self.turn ^= 1
        return out

    def run(self, plan_: Plan, q, k_pages, v_pages, kv_indptr, kv_indices,
            kv_last_page_len, sm_scale, out=None, lse=None, stream=None,
            phase: str = "both"):
        return run(plan_, q, k_pages, v_pages, kv_indptr, kv_indices,
                   kv_last_page_len, self.int_ws, self.float_ws, sm_scale,
                   out=out, lse=lse, stream=stream, phase=phase)
