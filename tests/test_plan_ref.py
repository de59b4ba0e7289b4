"""Invariants of the plain-Python split-KV planning rule (oracle.plan_ref).

The rule is this library's design (the pages fix only that planning reads
lengths and page-table metadata and prepares a schedule, "FlashInfer"
(aiwiki.ai/wiki/flashinfer), "Plan and run"), so it is pinned by what any
correct split-KV schedule must satisfy: the units of a request tile
[0, L_b) exactly, CTAs get contiguous, balanced shares, every request gets at
least min(m, n_b) pieces, and partial slots match the merge lists.
"""
import numpy as np
import pytest

from oracle import plan_ref

HEADER = plan_ref.HEADER_WORDS


def decode_image(img):
    img = [int(x) for x in img]
    hdr = img[:HEADER]
    batch, ctas, nunits, nslots, nsplit = hdr[2], hdr[3], hdr[4], hdr[5], hdr[6]
    off = HEADER
    cta_ptr = img[off:off + ctas + 1]
    off += ctas + 1
    units = [tuple(img[off + 4 * i: off + 4 * i + 4]) for i in range(nunits)]
    off += 4 * nunits
    merge_indptr = img[off:off + nsplit + 1]
    off += nsplit + 1
    merge_req = img[off:off + nsplit]
    off += nsplit
    assert off == len(img)
    return hdr, cta_ptr, units, merge_indptr, merge_req


def random_table(rng, batch, page_size, max_len, empty_frac=0.1):
    lengths = rng.integers(1, max_len + 1, size=batch)
    lengths[rng.random(batch) < empty_frac] = 0
    npages = (lengths + page_size - 1) // page_size
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    last = np.where(npages > 0, lengths - (npages - 1) * page_size, 0).astype(np.int32)
    return lengths, indptr, last


CASES = [
    # batch, page_size, max_len, tile, ctas, min_chunks
    (1, 16, 512, 16, 152, 1),
    (64, 16, 4096, 16, 152, 1),
    (256, 1, 5000, 16, 152, 1),
    (8, 64, 131072, 16, 152, 132),
    (5, 3, 40, 16, 4, 1),
    (17, 7, 300, 32, 9, 3),
    (3, 1, 2, 128, 152, 1),
    (40, 16, 100, 16, 1, 1),
    (12, 2, 1000, 64, 7, 5),
]


@pytest.mark.parametrize("case", CASES)
def test_plan_invariants(case):
    batch, page_size, max_len, tile, ctas, m = case
    rng = np.random.default_rng(hash(case) % (2 ** 32))
    lengths, indptr, last = random_table(rng, batch, page_size, max_len)
    img = plan_ref.plan_image(indptr, last, page_size=page_size, tile_tokens=tile,
                              num_ctas=ctas, min_chunks=m, num_qo_heads=32)
    assert img.dtype == np.int32
    hdr, cta_ptr, units, merge_indptr, merge_req = decode_image(img)
    assert hdr[0] == plan_ref.MAGIC and hdr[1] == plan_ref.LAYOUT_VERSION
    assert hdr[2] == batch and hdr[3] == ctas and hdr[7] == tile
    assert hdr[8] == page_size and hdr[11] == m and hdr[12] == 0 and hdr[13] == 32
    tiles = [(int(n) + tile - 1) // tile for n in lengths]
    assert hdr[9] == sum(tiles)
    quota = hdr[10]
    assert quota == max(1, -(-sum(tiles) // ctas))

    # CTA ranges are contiguous and cover all units, each within its quota
    assert cta_ptr[0] == 0 and cta_ptr[-1] == len(units)
    assert all(a <= b for a, b in zip(cta_ptr, cta_ptr[1:]))
    for c in range(ctas):
        work = sum(-(-(u[2] - u[1]) // tile) for u in units[cta_ptr[c]:cta_ptr[c + 1]])
        assert work <= quota

    # units of each request tile [0, L_b) exactly, in order
    by_req = {}
    for req, t0, t1, slot in units:
        by_req.setdefault(req, []).append((t0, t1, slot))
    assert sorted(by_req) == list(range(batch))
    next_slot = 0
    for b in range(batch):
        pieces = by_req[b]
        if lengths[b] == 0:
            assert pieces == [(0, 0, -1)]
            continue
        assert pieces[0][0] == 0 and pieces[-1][1] == lengths[b]
        for (a0, a1, _), (b0, _, _) in zip(pieces, pieces[1:]):
            assert a1 == b0 and a0 < a1
        assert all(t0 % tile == 0 for t0, _, _ in pieces)
        assert len(pieces) >= min(m, tiles[b])
        if len(pieces) == 1:
            assert pieces[0][2] == -1
        else:
            slots = [s for _, _, s in pieces]
            assert slots == list(range(next_slot, next_slot + len(pieces)))
            next_slot += len(pieces)
    assert next_slot == hdr[5]

    # merge lists name exactly the split requests, with their slot ranges
    split = [b for b in range(batch) if len(by_req[b]) > 1]
    assert merge_req == split
    assert merge_indptr[0] == 0
    for i, b in enumerate(split):
        assert merge_indptr[i + 1] - merge_indptr[i] == len(by_req[b])


def test_long_context_reading_gives_at_least_132_partitions_per_request():
    lengths = [131072] * 8
    indptr = np.arange(9, dtype=np.int32) * 2048
    last = np.full(8, 64, dtype=np.int32)
    img = plan_ref.plan_image(indptr, last, page_size=64, tile_tokens=16,
                              num_ctas=152, min_chunks=132, num_qo_heads=64)
    _, _, units, merge_indptr, merge_req = decode_image(img)
    assert merge_req == list(range(8))
    for i in range(8):
        assert merge_indptr[i + 1] - merge_indptr[i] >= 132
    assert sum(u[2] - u[1] for u in units) == sum(lengths)


def test_all_empty_batch():
    img = plan_ref.plan_image(np.zeros(4, np.int32), np.zeros(3, np.int32),
                              page_size=16, tile_tokens=16, num_ctas=8,
                              min_chunks=1, num_qo_heads=8)
    hdr, cta_ptr, units, merge_indptr, merge_req = decode_image(img)
    assert units == [(0, 0, 0, -1), (1, 0, 0, -1), (2, 0, 0, -1)]
    assert cta_ptr == [0] + [3] * 8 and merge_req == [] and merge_indptr == [0]


def test_zero_batch():
    img = plan_ref.plan_image(np.zeros(1, np.int32), np.zeros(0, np.int32),
                              page_size=16, tile_tokens=16, num_ctas=2,
                              min_chunks=1, num_qo_heads=8)
    hdr, cta_ptr, units, _, _ = decode_image(img)
    assert units == [] and cta_ptr == [0, 0, 0]
