"""Plain-Python statement of the split-KV planning rule: TEST INFRASTRUCTURE ONLY.

The pages fix only that planning looks at sequence lengths and page-table
metadata, chooses a schedule and prepares workspace data that a later run
applies ("FlashInfer" (aiwiki.ai/wiki/flashinfer), "Plan and run"), and that a
long cache may be split across GPU work units whose partial states are merged
afterwards (same page, "Attention states").  The concrete rule below is this
library's own design; it is integer-only and deterministic so that the
library's C++ planner can be checked against it bit for bit.

Rule ("balanced contiguous split"), with T = tile_tokens, C = num_ctas and
m = min_chunks_per_request:

1. Request b has npages_b = indptr[b+1] - indptr[b] pages and
   L_b = 0 if npages_b == 0 else (npages_b - 1) * P + last_page_len[b] tokens,
   i.e. n_b = ceil(L_b / T) tiles.
2. Cap-chunk size c_b = n_b when m == 1, else max(1, floor(n_b / m)) tiles;
   request b is first cut at tile multiples of c_b (so it has at least
   min(m, n_b) pieces).
3. W = sum n_b, per-CTA quota Q = max(1, ceil(W / C)) tiles.
4. Requests are walked in order and their tiles dealt to CTAs 0, 1, ... in
   order, each CTA taking Q tiles (the last one takes whatever remains).  A
   piece ends at a cap-chunk boundary, at the end of the CTA's quota, or at the
   end of the request.  Each piece is one unit (req, tok_begin, tok_end) with
   tok_end clipped to L_b.  An empty request is one unit (b, 0, 0) in the
   current CTA and uses no quota.
5. A request with a single unit writes its final output directly
   (partial = -1).  Otherwise its units get consecutive partial slots in
   emission order, and the request is listed for the merge step.

Plan image (int32 words):
  [0] magic 0x31444B50  [1] layout version 1  [2] B  [3] C  [4] units U
  [5] partial slots S  [6] split requests R  [7] T  [8] P  [9] W  [10] Q
  [11] m  [12] device status (0)  [13] Hq  [14] 0  [15] 0
  then cta_unit_ptr[C + 1], units[U][4] = (req, tok_begin, tok_end, partial),
  merge_indptr[R + 1] (slot ranges), merge_req[R].
"""
from __future__ import annotations

import numpy as np

MAGIC = 0x31444B50
LAYOUT_VERSION = 1
HEADER_WORDS = 16


def request_lengths(kv_indptr, kv_last_page_len, page_size):
    """Tokens per request under the CSR reading (full pages but the last)."""
    lengths = []
    for b in range(len(kv_last_page_len)):
        npages = int(kv_indptr[b + 1]) - int(kv_indptr[b])
        if npages == 0:
            lengths.append(0)
        else:
            lengths.append((npages - 1) * page_size + int(kv_last_page_len[b]))
    return lengths


def ceil_div(a, b):
    return -(-a // b)


def plan_units(lengths, tile_tokens, num_ctas, min_chunks):
    """Steps 1-4: the CTA ranges and the (req, tok_begin, tok_end) units."""
    tiles = [ceil_div(length, tile_tokens) for length in lengths]
    total = sum(tiles)
    quota = max(1, ceil_div(total, num_ctas))
    units = []
    cta_ptr = [0]
    cta = 0
    used = 0
    for b, n in enumerate(tiles):
        if n == 0:
            units.append((b, 0, 0))
            continue
        cap = n if min_chunks <= 1 else max(1, n // min_chunks)
        pos = 0
        while pos < n:
            if used >= quota and cta < num_ctas - 1:
                cta_ptr.append(len(units))
                cta += 1
                used = 0
            room = quota - used if cta < num_ctas - 1 else n - pos
            take = min(n - pos, cap - pos % cap, room)
            units.append((b, pos * tile_tokens,
                          min((pos + take) * tile_tokens, lengths[b])))
            pos += take
            used += take
    while len(cta_ptr) < num_ctas + 1:
        cta_ptr.append(len(units))
    return cta_ptr, units, total, quota


def plan_image(kv_indptr, kv_last_page_len, *, page_size, tile_tokens,
               num_ctas, min_chunks, num_qo_heads):
    """The whole int32 plan image the library copies to the device."""
    lengths = request_lengths(kv_indptr, kv_last_page_len, page_size)
    batch = len(lengths)
    cta_ptr, units, total, quota = plan_units(lengths, tile_tokens, num_ctas,
                                              min_chunks)
    pieces = [0] * batch
    for req, _, _ in units:
        pieces[req] += 1
    rows = []
    slot = 0
    for req, t0, t1 in units:
        if pieces[req] == 1:
            rows.append((req, t0, t1, -1))
        else:
            rows.append((req, t0, t1, slot))
            slot += 1
    merge_indptr = [0]
    merge_req = []
    for b in range(batch):
        if pieces[b] > 1:
            merge_req.append(b)
            merge_indptr.append(merge_indptr[-1] + pieces[b])
    header = [MAGIC, LAYOUT_VERSION, batch, num_ctas, len(units), slot,
              len(merge_req), tile_tokens, page_size, total, quota,
              min_chunks, 0, num_qo_heads, 0, 0]
    words = list(header) + list(cta_ptr)
    for row in rows:
        words.extend(row)
    words.extend(merge_indptr)
    words.extend(merge_req)
    return np.array(words, dtype=np.int64).astype(np.int32)
