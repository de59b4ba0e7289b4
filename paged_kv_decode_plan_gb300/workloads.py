"""Seeded synthetic paged-KV decode inputs.

This module builds page tables and random query / key / value tensors and
nothing else: it holds none of the attention arithmetic, so that both the
CUDA path and the test oracle can consume the same inputs without sharing any
of the method.

Random values come from numpy's PCG64 generator.  Every tensor is produced in
fixed-size chunks, chunk j of tensor ``tag`` drawing from
``default_rng([seed, tag, j])``, so the result does not depend on the number
of threads used to fill it.  Values are standard normal in float32, optionally
scaled in float32, then rounded to half or bfloat16 (round to nearest even);
the rounded values are the inputs, so rounding is not an error of either side.

Draw order for a workload with seed s: request lengths from
``default_rng([s, 0])``, then the page permutation from ``default_rng([s, 1])``,
then q (tag 2), K (tag 3) and V (tag 4).

The five named workloads are the decode batches this library is measured on:

=========================  ===================================================
``single``                 1 request, 512 tokens, Hq 32 / Hkv 8, P 16, fp16,
                           32 pages taken in shuffled order from a 64-page pool
``batch64``                64 requests, lengths uniform on [128, 4096],
                           Hq 32 / Hkv 8, P 16, fp16, pages permuted over a
                           pool of exactly the pages used
``longtail``               256 requests, lengths round(exp(N(ln 1024, 1)))
                           clipped to [16, 32768], Hq 32 / Hkv 8, P 1, bf16
``cascade``                128 requests sharing one 8192-token prefix (512
                           pages stored once) plus suffixes uniform on
                           [64, 1024]; Hq 32 / Hkv 8, P 16, fp16
``longctx``                8 requests x 131072 tokens, Hq 64 / Hkv 8, P 64,
                           bf16, keys scaled by 0.5 before rounding
=========================  ===================================================
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

CHUNK_ELEMS = 1 << 20
HEAD_DIM = 128
TAG_LENGTHS, TAG_PERM, TAG_Q, TAG_K, TAG_V = 0, 1, 2, 3, 4

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class PageTable:
    """CSR page table: request b owns kv_indices[kv_indptr[b]:kv_indptr[b+1]]."""
    kv_indptr: np.ndarray          # int32 [B + 1]
    kv_indices: np.ndarray         # int32 [nnz]
    kv_last_page_len: np.ndarray   # int32 [B]
    page_size: int

    @property
    def batch(self) -> int:
        return int(self.kv_last_page_len.shape[0])

    def lengths(self) -> np.ndarray:
        npages = np.diff(self.kv_indptr.astype(np.int64))
        return np.where(npages > 0,
                        (npages - 1) * self.page_size + self.kv_last_page_len,
                        0).astype(np.int64)


@dataclass
class PagedBatch:
    """One decode batch: queries, the page pool and one or more tables."""
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                      # "f16" | "bf16"
    q: torch.Tensor                 # [B, Hq, D] CPU
    k_pages: torch.Tensor           # [num_pages, P, Hkv, D] CPU (NHD)
    v_pages: torch.Tensor
    table: PageTable                # the table attention is defined over
    sm_scale: float
    extra_tables: dict = field(default_factory=dict)   # e.g. cascade parts
    min_chunks_per_request: int = 1

    @property
    def batch(self) -> int:
        return self.table.batch

    @property
    def page_size(self) -> int:
        return self.table.page_size

    @property
    def num_pages(self) -> int:
        return int(self.k_pages.shape[0])

    def kv_bytes(self, table: PageTable | None = None) -> int:
        """Bytes of K and V the table's tokens occupy (2 tensors)."""
        t = self.table if table is None else table
        elem = self.k_pages.element_size()
        return int(t.lengths().sum()) * 2 * self.num_kv_heads * self.head_dim * elem


def _fill_normal(shape, dtype: str, seed: int, tag: int, scale: float = 1.0,
                 pin: bool = False, threads: int | None = None) -> torch.Tensor:
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=TORCH_DTYPES[dtype], pin_memory=pin)
    chunks = (n + CHUNK_ELEMS - 1) // CHUNK_ELEMS

    def work(j):
        lo = j * CHUNK_ELEMS
        hi = min(n, lo + CHUNK_ELEMS)
        x = np.random.default_rng([seed, tag, j]).standard_normal(
            hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[lo:hi] = torch.from_numpy(x).to(TORCH_DTYPES[dtype])

    workers = threads or min(32, os.cpu_count() or 1)
    if chunks == 1 or workers == 1:
        for j in range(chunks):
            work(j)
    else:
        with ThreadPoolExecutor(workers) as pool:
            list(pool.map(work, range(chunks)))
    return out.view(*shape)


def table_from_lengths(lengths, page_size: int, page_ids) -> PageTable:
    """Assigns page_ids in order to the requests' pages."""
    lengths = [int(x) for x in lengths]
    npages = [(length + page_size - 1) // page_size for length in lengths]
    indptr = np.zeros(len(lengths) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(npages)
    page_ids = np.asarray(page_ids, dtype=np.int64)
    if page_ids.size < indptr[-1]:
        raise ValueError("not enough pages")
    last = np.array([length - (n - 1) * page_size if n > 0 else 0
                     for length, n in zip(lengths, npages)], dtype=np.int32)
    return PageTable(indptr.astype(np.int32),
                     page_ids[: indptr[-1]].astype(np.int32), last, page_size)


def make_paged(name: str, lengths, *, num_qo_heads: int, num_kv_heads: int,
               page_size: int, dtype: str, seed: int, head_dim: int = HEAD_DIM,
               pool_pages: int | None = None, k_scale: float = 1.0,
               q_scale: float = 1.0, pin: bool = False,
               min_chunks_per_request: int = 1) -> PagedBatch:
    """A decode batch over a shuffled page pool.

    The pool holds ``pool_pages`` pages (default: exactly the pages used); the
    requests' pages are the first pages of one random permutation of the pool,
    so unused pool pages hold random values nobody should read.
    """
    lengths = [int(x) for x in lengths]
    used = sum((length + page_size - 1) // page_size for length in lengths)
    pool = used if pool_pages is None else int(pool_pages)
    if pool < used:
        raise ValueError("pool too small")
    perm = np.random.default_rng([seed, TAG_PERM]).permutation(max(pool, 1))
    table = table_from_lengths(lengths, page_size, perm[:used])
    batch = len(lengths)
    q = _fill_normal((batch, num_qo_heads, head_dim), dtype, seed, TAG_Q,
                     q_scale, pin)
    shape = (max(pool, 1), page_size, num_kv_heads, head_dim)
    k = _fill_normal(shape, dtype, seed, TAG_K, k_scale, pin)
    v = _fill_normal(shape, dtype, seed, TAG_V, 1.0, pin)
    return PagedBatch(name, num_qo_heads, num_kv_heads, head_dim, dtype, q, k,
                      v, table, 1.0 / math.sqrt(head_dim),
                      min_chunks_per_request=min_chunks_per_request)


def single(seed: int = 1001, pin: bool = False) -> PagedBatch:
    """1 request x 512 tokens, 32 of a 64-page pool, Hq 32 / Hkv 8, fp16."""
    return make_paged("single", [512], num_qo_heads=32, num_kv_heads=8,
                      page_size=16, dtype="f16", seed=seed, pool_pages=64,
                      pin=pin)


def batch64(seed: int = 1002, pin: bool = False) -> PagedBatch:
    """64 requests, lengths uniform on [128, 4096], P 16, fp16."""
    lengths = np.random.default_rng([seed, TAG_LENGTHS]).integers(
        128, 4096, size=64, endpoint=True)
    return make_paged("batch64", lengths, num_qo_heads=32, num_kv_heads=8,
                      page_size=16, dtype="f16", seed=seed, pin=pin)


def longtail_lengths(seed: int, batch: int = 256):
    z = np.random.default_rng([seed, TAG_LENGTHS]).standard_normal(batch)
    return np.clip(np.rint(np.exp(math.log(1024.0) + z)), 16, 32768).astype(np.int64)


def longtail(seed: int = 1003, pin: bool = False) -> PagedBatch:
    """256 requests, log-normal lengths (median 1024, sigma 1), P 1, bf16."""
    return make_paged("longtail", longtail_lengths(seed), num_qo_heads=32,
                      num_kv_heads=8, page_size=1, dtype="bf16", seed=seed,
                      pin=pin)


def cascade(seed: int = 1004, pin: bool = False, batch: int = 128,
            prefix_tokens: int = 8192, suffix_range=(64, 1024)) -> PagedBatch:
    """Shared-prefix batch: one prefix stored once, per-request suffixes.

    ``table`` is the combined prefix + suffix table (what attention is
    defined over); ``extra_tables`` holds ``prefix`` (every row lists the same
    prefix pages) and ``suffix`` (each request's own pages).
    """
    page_size = 16
    if prefix_tokens % page_size:
        raise ValueError("prefix must fill whole pages")
    suffix = np.random.default_rng([seed, TAG_LENGTHS]).integers(
        suffix_range[0], suffix_range[1], size=batch, endpoint=True)
    prefix_pages = prefix_tokens // page_size
    suffix_pages = int(sum((int(s) + page_size - 1) // page_size for s in suffix))
    pool = prefix_pages + suffix_pages
    perm = np.random.default_rng([seed, TAG_PERM]).permutation(pool)
    shared = perm[:prefix_pages]
    suffix_table = table_from_lengths(suffix, page_size, perm[prefix_pages:])
    prefix_table = PageTable(
        (np.arange(batch + 1, dtype=np.int64) * prefix_pages).astype(np.int32),
        np.tile(shared, batch).astype(np.int32),
        np.full(batch, page_size, dtype=np.int32), page_size)
    comb_indptr = prefix_table.kv_indptr.astype(np.int64) + suffix_table.kv_indptr
    comb_indices = np.concatenate([
        np.concatenate([shared, suffix_table.kv_indices[
            suffix_table.kv_indptr[b]:suffix_table.kv_indptr[b + 1]]])
        for b in range(batch)]).astype(np.int32)
    combined = PageTable(comb_indptr.astype(np.int32), comb_indices,
                         suffix_table.kv_last_page_len.copy(), page_size)
    q = _fill_normal((batch, 32, HEAD_DIM), "f16", seed, TAG_Q, 1.0, pin)
    shape = (pool, page_size, 8, HEAD_DIM)
    k = _fill_normal(shape, "f16", seed, TAG_K, 1.0, pin)
    v = _fill_normal(shape, "f16", seed, TAG_V, 1.0, pin)
    return PagedBatch("cascade", 32, 8, HEAD_DIM, "f16", q, k, v, combined,
                      1.0 / math.sqrt(HEAD_DIM),
                      extra_tables={"prefix": prefix_table, "suffix": suffix_table})


def longctx(seed: int = 1005, pin: bool = False, batch: int = 8,
            length: int = 131072) -> PagedBatch:
    """8 x 131072 tokens, Hq 64 / Hkv 8, P 64, bf16, keys x 0.5, >=132 splits."""
    return make_paged("longctx", [length] * batch, num_qo_heads=64,
                      num_kv_heads=8, page_size=64, dtype="bf16", seed=seed,
                      k_scale=0.5, pin=pin, min_chunks_per_request=132)


WORKLOADS = {"single": single, "batch64": batch64, "longtail": longtail,
             "cascade": cascade, "longctx": longctx}


def as_codes(t: torch.Tensor) -> np.ndarray:
    """16-bit storage codes of a half / bfloat16 CPU tensor, as numpy uint16."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("expected a 16-bit float tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
