"""The shared-prefix plan: its plain-Python restatement (oracle.prefix_plan_ref)
pinned by what the rule must guarantee, then the library's host planner
(pkd_plan_shared_prefix_host) compared with it bit for bit.

What pins the restatement, independent of both implementations: the pieces
tile the prefix [0, L) in 64-token steps with no gap or overlap, every piece
is non-empty and at most chunk_tiles steps long; the blocks fit the budget
(Hkv x row_tiles x chunks <= C) unless one piece is all there is; one more
piece of equal size would not fit or there are no steps left to give it; the
row tiles cover the batch x g query rows with less than one tile to spare;
the image holds the header fields and the page ids in order ("FlashInfer"
(aiwiki.ai/wiki/flashinfer), "Plan and run", "Attention states").
"""
import inspect
import types

import numpy as np
import pytest

import oracle.prefix_plan_ref as original
import paged_kv_decode_plan_gb300 as pkd

ref = original


def ceil_div(a, b):
    return -(-a // b)


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 3, 4, 6, 8, 12, 16]))
        page = int(rng.choice([16, 32, 64]))
        npages = int(rng.choice([0, 1, 2, 5, 33, 512, 1500]))
        last = int(rng.integers(1, page + 1))
        batch = int(rng.choice([0, 1, 2, 7, 63, 64, 65, 128, 300]))
        ctas = int(rng.choice([1, 2, 7, 8, 48, 104, 148, 152, 1000]))
        pool = npages + int(rng.integers(1, 50))
        pages = rng.permutation(pool)[:npages]
        yield dict(batch=batch, hq=hkv * g, hkv=hkv, page=page, pages=pages, last=last,
                   ctas=ctas, pool=pool)


def check_rule(c):
    s, img = ref.plan(c["batch"], c["hq"], c["hkv"], c["page"], c["pages"], c["last"],
                      c["ctas"])
    n = len(c["pages"])
    length = 0 if n == 0 else (n - 1) * c["page"] + c["last"]
    assert s["prefix_len"] == length
    steps = ceil_div(length, 64)
    chunks, ct, rt = s["chunks"], s["chunk_tiles"], s["row_tiles"]
    assert chunks >= 1
    # the pieces tile [0, L) in 64-token steps, each non-empty (when L > 0)
    ranges = ref.chunk_ranges(length, chunks, ct)
    assert len(ranges) == chunks
    pos = 0
    for t0, t1 in ranges:
        assert t0 == pos and t0 % 64 == 0
        assert (t1 > t0) or length == 0
        assert t1 - t0 <= 64 * ct
        pos = t1
    assert pos == length
    # row tiles cover the rows with less than one tile to spare
    rows = c["batch"] * (c["hq"] // c["hkv"])
    assert rt * 256 >= rows and (rt - 1) * 256 < max(rows, 1)
    # blocks fit the budget unless one piece is all there is
    base = c["hkv"] * rt
    assert base * chunks <= c["ctas"] or chunks == 1
    assert s["num_blocks"] == base * chunks
    # no more pieces of equal size fit (or every step has its own piece)
    if steps > 0:
        assert chunks == steps or base * (chunks + 1) > c["ctas"] or \
            ceil_div(steps, ceil_div(steps, chunks + 1)) == chunks
        assert ct == ceil_div(steps, chunks) or ceil_div(steps, ct) == chunks
    # the image: header fields, then the page ids in order
    assert img.dtype == np.int32 and img.size == 16 + n
    assert list(img[:11]) == [0x50444B50, 1, c["batch"], c["hq"], c["hkv"], c["page"],
                              length, n, chunks, ct, rt]
    assert not img[11:16].any()
    assert np.array_equal(img[16:], np.asarray(c["pages"], np.int32))
    assert s["int_ws_bytes_used"] == 4 * img.size


def test_rule_invariants():
    for c in _cases(400, 0):
        check_rule(c)


def test_pieces_by_brute_force():
    # every (steps, budget) of a small grid: the chosen piece size is the
    # smallest size whose piece count fits the budget (capped at one piece
    # per step), found by trying all sizes
    for steps in range(1, 40):
        for ctas in range(1, 40):
            for hkv in (1, 2, 8):
                length = 64 * steps - 5
                pages = np.arange(ceil_div(length, 16))
                last = length - 16 * (pages.size - 1)
                s, _ = ref.plan(4, hkv * 2, hkv, 16, pages, last, ctas)
                fit = [k for k in range(1, steps + 1) if hkv * k <= ctas] or [1]
                size = ceil_div(steps, max(fit))
                assert s["chunk_tiles"] == size, (steps, ctas, hkv)
                assert s["chunks"] == ceil_div(steps, size)


MUTANTS = {
    "row tiles rounded down": ("max(1, ceil_div(batch * group, ROW_TILE))",
                               "max(1, batch * group // ROW_TILE)"),
    "budget ignores row tiles": ("num_ctas // (num_kv_heads * row_tiles)",
                                 "num_ctas // num_kv_heads"),
    "piece size rounded down": ("chunk_tiles = ceil_div(steps, wanted) if",
                                "chunk_tiles = max(1, steps // wanted) if"),
    "steps rounded down": ("steps = ceil_div(length, STEP_TOKENS)\n    wanted",
                           "steps = length // STEP_TOKENS\n    wanted"),
    "pieces not recounted": ("chunks = ceil_div(steps, chunk_tiles) if chunk_tiles > 0 else wanted",
                             "chunks = wanted"),
    "length counts the last page full": (
        "(num_pages - 1) * page_size + last_page_len", "num_pages * page_size"),
    "header swaps kv and q heads": ("image[3] = num_qo_heads\n    image[4] = num_kv_heads",
                                    "image[3] = num_kv_heads\n    image[4] = num_qo_heads"),
}


def _mutated(old, new):
    src = inspect.getsource(original)
    assert src.count(old) == 1, old
    mod = types.ModuleType("prefix_plan_ref_mutant")
    exec(compile(src.replace(old, new), "prefix_plan_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_planted_mistake_fails_a_pin(name, monkeypatch):
    monkeypatch.setitem(globals(), "ref", _mutated(*MUTANTS[name]))
    failed = 0
    for pin in (test_rule_invariants, test_pieces_by_brute_force):
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed += 1
    assert failed >= 1, name


def _problem(c):
    return pkd.make_problem(batch=c["batch"], num_qo_heads=c["hq"],
                            num_kv_heads=c["hkv"], page_size=c["page"], dtype="f16",
                            num_pages=c["pool"], num_ctas=c["ctas"])


def test_library_prefix_plan_is_bit_exact():
    for c in _cases(600, 1):
        plan, image = pkd.plan_shared_prefix_host(_problem(c), c["pages"], c["last"])
        s, ref_img = ref.plan(c["batch"], c["hq"], c["hkv"], c["page"], c["pages"],
                              c["last"], c["ctas"])
        assert image.tobytes() == ref_img.tobytes(), c
        for key, value in s.items():
            assert getattr(plan, key) == value, (key, c)
        assert plan.valid == 1


def test_library_prefix_plan_errors():
    c = next(_cases(1, 2))
    c.update(pages=np.array([0, 3, 5]), pool=6, last=4, page=16)
    bad = dict(c, pages=np.array([0, 6, 5]))
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_shared_prefix_host(_problem(bad), bad["pages"], bad["last"])
    assert e.value.status == -2
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_shared_prefix_host(_problem(c), c["pages"], 17)
    assert e.value.status == -2
    odd = dict(c, page=8)
    with pytest.raises(pkd.PkdError) as e:
        pkd.plan_shared_prefix_host(_problem(odd), odd["pages"], 4)
    assert e.value.status == -4
