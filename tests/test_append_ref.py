"""Pins of the page-append restatement (oracle.append_ref).

Appending writes through the page table, so the facts fixed outside it are:
each appended row reads back through the same table unchanged, rows not
appended are untouched, and the order of the new tokens does not matter.  The
HND branch is pinned to the NHD one: the two layouts hold the same values
with the slot and head axes exchanged ("Welcome to FlashInfer's
documentation!", "KV-Cache Layout in FlashInfer", "Layout: NHD/HND"), so
appending into HND pools must give, bit for bit, the HND transpose of
appending into the same NHD pools.
"""
import numpy as np

from oracle import append_ref


def _case(rng, lengths, page, hkv=2, d=8):
    npages = [(n + page - 1) // page for n in lengths]
    pool = sum(npages) + 3
    perm = rng.permutation(pool)
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    indices = perm[: sum(npages)].astype(np.int32)
    last = np.array([n - (k - 1) * page if k else 0 for n, k in zip(lengths, npages)],
                    np.int32)
    k = rng.standard_normal((pool, page, hkv, d)).astype(np.float32)
    v = rng.standard_normal((pool, page, hkv, d)).astype(np.float32)
    return k, v, indptr, indices, last


def test_appended_rows_read_back_and_others_are_untouched():
    rng = np.random.default_rng(0)
    lengths = [5, 17, 1, 0, 33]
    k, v, indptr, indices, last = _case(rng, lengths, 4)
    # the decode step: one new token per non-empty request, at its last slot
    bi = np.array([0, 1, 2, 4], np.int32)
    pos = np.array([4, 16, 0, 32], np.int32)
    kn = rng.standard_normal((4, 2, 8)).astype(np.float32)
    vn = rng.standard_normal((4, 2, 8)).astype(np.float32)
    k2, v2, skipped = append_ref.append_kv(k, v, kn, vn, bi, pos, indptr, indices, last)
    assert skipped == []
    for i, (b, t) in enumerate(zip(bi, pos)):
        rows_k = append_ref.gather_tokens(k2, indptr, indices, last, b)
        rows_v = append_ref.gather_tokens(v2, indptr, indices, last, b)
        assert np.array_equal(rows_k[t], kn[i]) and np.array_equal(rows_v[t], vn[i])
    changed = np.argwhere(np.any(k2 != k, axis=(2, 3)))
    assert len(changed) == 4  # exactly the four (page, slot) rows


def test_append_order_does_not_matter_and_out_of_range_is_skipped():
    rng = np.random.default_rng(1)
    lengths = [40, 9, 64]
    k, v, indptr, indices, last = _case(rng, lengths, 16)
    n = 30
    bi = rng.integers(0, 3, n).astype(np.int32)
    pos = np.array([rng.integers(0, lengths[b]) for b in bi], np.int32)
    # distinct (request, position) pairs so the order cannot matter
    _, keep = np.unique(bi.astype(np.int64) * 1000 + pos, return_index=True)
    bi, pos = bi[keep], pos[keep]
    kn = rng.standard_normal((bi.size, 2, 8)).astype(np.float32)
    vn = rng.standard_normal((bi.size, 2, 8)).astype(np.float32)
    a = append_ref.append_kv(k, v, kn, vn, bi, pos, indptr, indices, last)
    p = rng.permutation(bi.size)
    b2 = append_ref.append_kv(k, v, kn[p], vn[p], bi[p], pos[p], indptr, indices, last)
    assert np.array_equal(a[0], b2[0]) and np.array_equal(a[1], b2[1])
    bad_bi = np.array([0, 1, 5, -1], np.int32)
    bad_pos = np.array([40, 3, 0, 0], np.int32)  # past the end, ok, no request x2
    _, _, skipped = append_ref.append_kv(k, v, kn[:4], vn[:4], bad_bi, bad_pos,
                                         indptr, indices, last)
    assert skipped == [0, 2, 3]


def test_appended_token_is_what_its_request_attends_to():
    # Pinned through the attention oracle's own page-table walk (ref_attn.c,
    # pinned against brute force): a new key that outscores every other key
    # of its request by > 100 makes attention over the request return the new
    # value; requests that received nothing are not pulled toward it.
    import math
    import oracle
    rng = np.random.default_rng(2)
    lengths = [5, 17, 1, 33, 9]
    page, hkv, g, d = 4, 2, 2, 8
    k, v, indptr, indices, last = _case(rng, lengths, page, hkv, d)
    q = np.repeat(rng.standard_normal((len(lengths), hkv, 1, d)), g, axis=2)
    q = q.reshape(len(lengths), hkv * g, d)           # the group's query heads agree
    bi = np.array([0, 1, 2, 3], np.int32)
    pos = np.array([4, 16, 0, 32], np.int32)           # each request's last slot
    kn = 40.0 * q[bi][:, ::g, :]                        # [new token, Hkv, D]
    vn = rng.standard_normal((bi.size, hkv, d))
    k2, v2, skipped = append_ref.append_kv(k.astype(np.float64), v.astype(np.float64), kn, vn,
                                           bi, pos, indptr, indices, last)
    assert skipped == []
    out, _ = oracle.decode(q, k2, v2, indptr, indices, last, dtype="f64",
                           sm_scale=1.0 / math.sqrt(d))
    out = out.reshape(len(lengths), hkv * g, d)
    for i, b in enumerate(bi):
        for h in range(hkv * g):
            assert np.max(np.abs(out[b, h] - vn[i, h // g])) <= 1e-12
    for h in range(hkv * g):   # request 4 got no token
        assert min(np.max(np.abs(out[4, h] - vn[i, h // g])) for i in range(bi.size)) > 0.1


def _hnd(x):
    """NHD [pages, P, Hkv, D] -> HND [pages, Hkv, P, D] (the same values)."""
    return np.ascontiguousarray(np.swapaxes(x, 1, 2))


def test_hnd_append_is_the_transpose_of_nhd_append():
    # page sizes above, equal to and below Hkv, so a slot / head mix-up
    # cannot hide behind equal axis lengths
    for seed, (lengths, page, hkv) in enumerate([([5, 17, 1, 0, 33], 4, 2),
                                                 ([40, 9, 64], 16, 4),
                                                 ([7, 12, 3], 3, 3),
                                                 ([9, 2], 1, 8)]):
        rng = np.random.default_rng(100 + seed)
        k, v, indptr, indices, last = _case(rng, lengths, page, hkv)
        n = 12
        bi = rng.integers(0, len(lengths), n).astype(np.int32)
        pos = np.array([rng.integers(0, max(lengths[b], 1)) for b in bi], np.int32)
        pos[0] = 10_000   # one token past its request's end: skipped either way
        _, keep = np.unique(bi.astype(np.int64) * 100_000 + pos, return_index=True)
        bi, pos = bi[keep], pos[keep]
        kn = rng.standard_normal((bi.size, hkv, 8)).astype(np.float32)
        vn = rng.standard_normal((bi.size, hkv, 8)).astype(np.float32)
        k_nhd, v_nhd, skip_nhd = append_ref.append_kv(k, v, kn, vn, bi, pos, indptr,
                                                      indices, last)
        k_hnd, v_hnd, skip_hnd = append_ref.append_kv(_hnd(k), _hnd(v), kn, vn, bi, pos,
                                                      indptr, indices, last, layout="HND")
        assert skip_hnd == skip_nhd and len(skip_nhd) >= 1
        assert k_hnd.shape == _hnd(k).shape
        assert np.array_equal(k_hnd, _hnd(k_nhd)) and np.array_equal(v_hnd, _hnd(v_nhd))
