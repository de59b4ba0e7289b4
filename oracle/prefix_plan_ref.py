"""Plain-Python statement of the shared-prefix planning rule: TEST
INFRASTRUCTURE ONLY.

The pages fix that a prefix shared by many requests is evaluated separately
from the requests' own suffixes and the two partial states are merged by
their log-sum-exp values ("FlashInfer" (aiwiki.ai/wiki/flashinfer), "Attention
states"), and that planning reads lengths and metadata and prepares workspace
data for a later run (same page, "Plan and run").  How the prefix work is cut
into pieces is this library's own design; the rule is integer-only and
deterministic so that the library's planner can be checked against it bit for
bit.

Rule, for B requests, Hq query heads, Hkv key/value heads (g = Hq / Hkv), page
size P, a prefix of n pages whose last page holds `last` tokens, and a budget
of C blocks:

1. The prefix has L = 0 tokens if n == 0, else (n - 1) * P + last.
2. Per key/value head the queries form one dense tile of B * g rows, cut into
   row_tiles = max(1, ceil(B * g / 256)) tiles of 256 rows.
3. The prefix is walked in steps of 64 tokens: T = ceil(L / 64) steps.
4. chunks0 = max(1, min(T, floor(C / (Hkv * row_tiles)))) pieces are wanted;
   each piece takes chunk_tiles = ceil(T / chunks0) steps (0 when T == 0), and
   the pieces actually used are chunks = ceil(T / chunk_tiles) (chunks0 when
   T == 0).  Piece c covers steps [c * chunk_tiles, min((c + 1) * chunk_tiles,
   T)).
5. One block per (key/value head, row tile, piece): Hkv * row_tiles * chunks
   blocks; every (request, query head, piece) leaves one fp32 state.

Plan image (int32 words): a 16-word header
  [0] magic 0x50444B50  [1] version 1  [2] B  [3] Hq  [4] Hkv  [5] P  [6] L
  [7] n  [8] chunks  [9] chunk_tiles  [10] row_tiles  [11] 0  [12] device
  status (0)  [13..15] 0
followed by the n prefix page ids in order.
"""
from __future__ import annotations

import numpy as np

MAGIC = 0x50444B50
VERSION = 1
HEADER_WORDS = 16
STEP_TOKENS = 64      # tokens per step of the prefix walk
ROW_TILE = 256        # query rows per block


def ceil_div(a, b):
    return -(-a // b)


def prefix_length(num_pages, last_page_len, page_size):
    """Tokens of a prefix stored as num_pages pages (all full but the last)."""
    return 0 if num_pages == 0 else (num_pages - 1) * page_size + last_page_len


def split(batch, num_qo_heads, num_kv_heads, length, num_ctas):
    """(chunks, chunk_tiles, row_tiles) of the rule above."""
    group = num_qo_heads // num_kv_heads
    row_tiles = max(1, ceil_div(batch * group, ROW_TILE))
    steps = ceil_div(length, STEP_TOKENS)
    wanted = max(1, min(steps, num_ctas // (num_kv_heads * row_tiles)))
    chunk_tiles = ceil_div(steps, wanted) if steps > 0 else 0
    chunks = ceil_div(steps, chunk_tiles) if chunk_tiles > 0 else wanted
    return chunks, chunk_tiles, row_tiles


def chunk_ranges(length, chunks, chunk_tiles):
    """Token range [t0, t1) of each piece."""
    steps = ceil_div(length, STEP_TOKENS)
    out = []
    for c in range(chunks):
        s0 = min(c * chunk_tiles, steps)
        s1 = min((c + 1) * chunk_tiles, steps)
        out.append((min(s0 * STEP_TOKENS, length), min(s1 * STEP_TOKENS, length)))
    return out


def state_floats(num_qo_heads, head_dim=128):
    """Floats of one fp32 state slot: o [Hq][D], then lse [Hq] padded to a
    multiple of 4 floats."""
    return num_qo_heads * head_dim + ceil_div(num_qo_heads, 4) * 4


def plan(batch, num_qo_heads, num_kv_heads, page_size, pages, last_page_len, num_ctas):
    """Plan scalars (a dict) and the plan image (int32 array) for one prefix."""
    pages = [int(p) for p in pages]
    n = len(pages)
    length = prefix_length(n, int(last_page_len), page_size)
    chunks, chunk_tiles, row_tiles = split(batch, num_qo_heads, num_kv_heads, length,
                                           num_ctas)
    image = np.zeros(HEADER_WORDS + n, dtype=np.int32)
    image[0] = MAGIC
    image[1] = VERSION
    image[2] = batch
    image[3] = num_qo_heads
    image[4] = num_kv_heads
    image[5] = page_size
    image[6] = length
    image[7] = n
    image[8] = chunks
    image[9] = chunk_tiles
    image[10] = row_tiles
    image[HEADER_WORDS:] = pages
    scalars = {"prefix_len": length, "prefix_num_pages": n, "chunks": chunks,
               "chunk_tiles": chunk_tiles, "row_tiles": row_tiles,
               "num_blocks": num_kv_heads * row_tiles * chunks,
               "int_ws_bytes_used": 4 * (HEADER_WORDS + n),
               "float_ws_bytes_needed": 4 * batch * chunks * state_floats(num_qo_heads)}
    return scalars, image
