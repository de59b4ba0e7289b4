"""Oracle for paged decode attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports it and
shares no code with it.

* :func:`decode` and :func:`merge` call the plain fp64 C code in
  ``ref_attn.c`` (built with gcc by :func:`build`).
* :mod:`oracle.plan_ref` restates the split-KV work-list rule in plain Python.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(brute force against a library attention routine, closed forms, the union
property of merged states, permutation and shift invariance, empty rows), and
``tests/test_oracle_mutants.py`` shows that planted mistakes in a copy of
``ref_attn.c`` fail those pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ref_attn.c")
_LIB = os.path.join(_HERE, "libpkd_oracle.so")

F16, BF16, F32, F64 = 0, 1, 2, 3
_DTYPE_CODES = {"f16": F16, "float16": F16, "bf16": BF16, "bfloat16": BF16,
                "f32": F32, "float32": F32, "f64": F64, "float64": F64}


class OracleError(RuntimeError):
    pass


def compile_source(src: str, out: str) -> str:
    """gcc-compile one copy of the oracle C source into ``out``."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _native(path: str) -> bool:
    """True when the ELF file's machine field matches this host."""
    import platform
    want = {"x86_64": 62, "aarch64": 183}.get(platform.machine())
    with open(path, "rb") as f:
        head = f.read(20)
    return want is None or (len(head) == 20 and
                            int.from_bytes(head[18:20], "little") == want)


def build(force: bool = False) -> str:
    """Compile ``ref_attn.c`` into ``libpkd_oracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB) and _native(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(SOURCE)):
        return _LIB
    return compile_source(SOURCE, _LIB)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _raw(a: np.ndarray, dtype: str) -> np.ndarray:
    """Element storage for the C side: 16-bit codes for f16/bf16."""
    code = _DTYPE_CODES[dtype]
    if code in (F16, BF16):
        if a.dtype == np.float16:
            a = a.view(np.uint16)
        if a.dtype not in (np.uint16, np.int16):
            raise TypeError("f16/bf16 inputs are passed as 16-bit codes")
        return np.ascontiguousarray(a).view(np.uint16)
    want = np.float32 if code == F32 else np.float64
    return np.ascontiguousarray(a, dtype=want)


class Oracle:
    """ctypes view of one compiled copy of ``ref_attn.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        f64p = ctypes.POINTER(ctypes.c_double)
        vp = ctypes.c_void_p
        lib.orc_decode.restype = ctypes.c_int
        lib.orc_decode.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int64, i32p, i32p, i32p,
            ctypes.c_double, i64p, ctypes.c_int64, f64p, f64p]
        lib.orc_merge.restype = ctypes.c_int
        lib.orc_merge.argtypes = [ctypes.c_int64, ctypes.c_int, f64p, f64p,
                                  f64p, f64p, f64p, f64p]
        lib.orc_num_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def num_threads(self) -> int:
        """Threads the oracle's OpenMP loop uses."""
        return int(self.lib.orc_num_threads())

    def decode(self, q, k_pages, v_pages, kv_indptr, kv_indices,
               kv_last_page_len, *, dtype: str, sm_scale: float, rows=None,
               layout: str = "NHD"):
        """fp64 paged decode attention (page-table walk, two-pass softmax).

        q: [B, Hq, D]; k_pages, v_pages: [num_pages, P, Hkv, D] (NHD) or
        [num_pages, Hkv, P, D] (HND).  For f16 / bf16 the arrays hold the
        16-bit codes.  ``rows`` optionally lists flattened row ids b * Hq + h.
        Returns (out [n, D] float64, lse [n] float64), n = len(rows) or B * Hq.
        """
        if q.ndim != 3 or k_pages.ndim != 4 or v_pages.shape != k_pages.shape:
            raise ValueError("bad tensor ranks / shapes")
        batch, hq, d = q.shape
        if layout == "HND":
            num_pages, hkv, page_size, d2 = k_pages.shape
        elif layout == "NHD":
            num_pages, page_size, hkv, d2 = k_pages.shape
        else:
            raise ValueError("layout must be NHD or HND")
        if d2 != d:
            raise ValueError("head_dim mismatch")
        qr, kr, vr = _raw(q, dtype), _raw(k_pages, dtype), _raw(v_pages, dtype)
        indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
        indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
        last = np.ascontiguousarray(kv_last_page_len, dtype=np.int32)
        if indptr.shape != (batch + 1,) or last.shape != (batch,):
            raise ValueError("page-table shapes")
        if rows is None:
            n = batch * hq
            rows_p = None
        else:
            rows_a = np.ascontiguousarray(rows, dtype=np.int64)
            n = rows_a.size
            rows_p = _ptr(rows_a, ctypes.c_int64)
        out = np.zeros((n, d), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        if indices.size == 0:
            indices = np.zeros((1,), dtype=np.int32)
        rc = self.lib.orc_decode(
            batch, hq, hkv, d, page_size, _DTYPE_CODES[dtype],
            1 if layout == "HND" else 0, qr.ctypes.data,
            kr.ctypes.data, vr.ctypes.data, num_pages,
            _ptr(indptr, ctypes.c_int32), _ptr(indices, ctypes.c_int32),
            _ptr(last, ctypes.c_int32), float(sm_scale), rows_p, n,
            _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
        if rc != 0:
            raise OracleError("orc_decode failed with code %d" % rc)
        return out, lse

    def merge(self, v_a, s_a, v_b, s_b):
        """fp64 merge of two attention states; v: [..., D], s: [...]."""
        v_a = np.ascontiguousarray(v_a, dtype=np.float64)
        v_b = np.ascontiguousarray(v_b, dtype=np.float64)
        s_a = np.ascontiguousarray(s_a, dtype=np.float64)
        s_b = np.ascontiguousarray(s_b, dtype=np.float64)
        if v_a.shape != v_b.shape or s_a.shape != s_b.shape \
                or v_a.shape[:-1] != s_a.shape:
            raise ValueError("state shapes")
        d = v_a.shape[-1]
        n = int(np.prod(s_a.shape)) if s_a.ndim else 1
        v = np.zeros_like(v_a)
        s = np.zeros_like(s_a)
        rc = self.lib.orc_merge(
            n, d, _ptr(v_a, ctypes.c_double), _ptr(s_a, ctypes.c_double),
            _ptr(v_b, ctypes.c_double), _ptr(s_b, ctypes.c_double),
            _ptr(v, ctypes.c_double), _ptr(s, ctypes.c_double))
        if rc != 0:
            raise OracleError("orc_merge failed with code %d" % rc)
        return v, s


_default = None


def default() -> Oracle:
    """The oracle built from ``ref_attn.c`` as committed."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def decode(*args, **kwargs):
    return default().decode(*args, **kwargs)


def merge(*args, **kwargs):
    return default().merge(*args, **kwargs)


def num_threads() -> int:
    return default().num_threads()
