"""Page append restated in plain Python: TEST INFRASTRUCTURE ONLY.

"Welcome to FlashInfer's documentation!" (docs.flashinfer.ai), flashinfer.page
"Append new K/V tensors to Paged KV-Cache" (a title only).  Reading: new token
i belongs to request ``batch_indices[i]`` at position ``positions[i]`` of that
request; the page table already covers the request's new length; the token's
key and value rows (all heads) go to page ``kv_indices[kv_indptr[b] + t // P]``,
slot ``t % P`` of the NHD page tensors ([pages][P][Hkv][D]), or of the HND
ones ([pages][Hkv][P][D], "KV-Cache Layout in FlashInfer", "Layout:
NHD/HND").  Pinned by tests/test_append_ref.py: every appended token reads
back through the page table unchanged, the result does not depend on the
order of the new tokens, and appending into HND pools gives exactly the HND
transpose of appending into the same NHD pools.
"""
from __future__ import annotations

import numpy as np


def request_lengths(kv_indptr, kv_last_page_len, page_size):
    out = []
    for b in range(len(kv_last_page_len)):
        n = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        out.append(0 if n == 0 else (n - 1) * page_size + int(kv_last_page_len[b]))
    return out


def append_kv(k_pages, v_pages, k_new, v_new, batch_indices, positions, kv_indptr,
              kv_indices, kv_last_page_len, layout="NHD"):
    """Writes new rows into copies of the page tensors; returns the copies.

    k_pages / v_pages: [num_pages, P, Hkv, D] arrays (any dtype, copied);
    k_new / v_new: [n, Hkv, D].  Tokens outside their request's length or on
    a page id outside the pool are skipped and reported in the second return
    value (their indices).
    """
    k = np.array(k_pages, copy=True)
    v = np.array(v_pages, copy=True)
    num_pages = k.shape[0]
    page_size = k.shape[2] if layout == "HND" else k.shape[1]
    lengths = request_lengths(kv_indptr, kv_last_page_len, page_size)
    skipped = []
    for i in range(len(batch_indices)):
        b = int(batch_indices[i])
        t = int(positions[i])
        if b < 0 or b >= len(lengths) or t < 0 or t >= lengths[b]:
            skipped.append(i)
            continue
        page = int(kv_indices[int(kv_indptr[b]) + t // page_size])
        if page < 0 or page >= num_pages:
            skipped.append(i)
            continue
        if layout == "HND":
            k[page, :, t % page_size] = k_new[i]
            v[page, :, t % page_size] = v_new[i]
        else:
            k[page, t % page_size] = k_new[i]
            v[page, t % page_size] = v_new[i]
    return k, v, skipped


def gather_tokens(pages, kv_indptr, kv_indices, kv_last_page_len, b):
    """[L_b, Hkv, D] rows of request b read back through the page table."""
    page_size = pages.shape[1]
    n = request_lengths(kv_indptr, kv_last_page_len, page_size)[b]
    rows = [pages[int(kv_indices[int(kv_indptr[b]) + t // page_size]), t % page_size]
            for t in range(n)]
    return np.stack(rows) if rows else np.zeros((0,) + pages.shape[2:], pages.dtype)
