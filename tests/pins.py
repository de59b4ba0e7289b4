"""Checks that pin the fp64 oracle to facts fixed outside itself.

Each ``check_*`` takes an :class:`oracle.Oracle` and raises AssertionError when
the oracle disagrees with:

* a library attention routine (torch's scaled_dot_product_attention and
  scipy's logsumexp, both in float64) on tiny dense copies of paged inputs;
* closed forms: a single key returns its value vector; identical keys return
  the mean of the values with lse = s + ln n; a hand-checked grouped-head case;
* the union property of attention states ("FlashInfer"
  (aiwiki.ai/wiki/flashinfer), "Attention states"): merging the states of
  disjoint page sets equals attention over their union, in any grouping;
* invariances: permuting the page pool together with the page ids changes
  nothing; adding the same large negative constant to every logit (all logits
  below -5e4) leaves the output unchanged and shifts lse by that constant
  (same page, "Extreme-negative-logit correction");
* the empty-row rule (same section): no tokens gives (0, -inf), and such a
  state is the identity of the merge.

The inputs are tiny and exactly representable, so the bounds are near fp64
rounding.
"""
from __future__ import annotations

import math

import numpy as np
import scipy.special
import torch

F = torch.nn.functional


def _codes_and_values(x32: np.ndarray, dtype: str):
    """Round float32 values to f16/bf16; return (codes, exact float64)."""
    if dtype == "f16":
        h = x32.astype(np.float16)
        return h.view(np.uint16), h.astype(np.float64)
    t = torch.from_numpy(np.ascontiguousarray(x32)).to(torch.bfloat16)
    return (t.view(torch.int16).numpy().view(np.uint16),
            t.to(torch.float64).numpy())


def paged_case(rng, lengths, hq, hkv, d, p, dtype, extra_pages=2, scale_k=1.0):
    """Random paged batch; returns dict of codes, float64 copies and table."""
    npages = [(n + p - 1) // p for n in lengths]
    used = sum(npages)
    pool = used + extra_pages
    perm = rng.permutation(pool)
    indptr = np.concatenate([[0], np.cumsum(npages)]).astype(np.int32)
    indices = perm[:used].astype(np.int32)
    last = np.array([n - (k - 1) * p if k else 0
                     for n, k in zip(lengths, npages)], dtype=np.int32)
    q32 = rng.standard_normal((len(lengths), hq, d)).astype(np.float32)
    k32 = (rng.standard_normal((pool, p, hkv, d)) * scale_k).astype(np.float32)
    v32 = rng.standard_normal((pool, p, hkv, d)).astype(np.float32)
    case = dict(lengths=list(lengths), hq=hq, hkv=hkv, d=d, p=p, dtype=dtype,
                indptr=indptr, indices=indices, last=last)
    for name, x in (("q", q32), ("k", k32), ("v", v32)):
        codes, vals = _codes_and_values(x, dtype)
        case[name] = codes
        case[name + "64"] = vals
    case["sm_scale"] = 1.0 / math.sqrt(d)
    return case


def run_case(orc, case, rows=None, indptr=None, indices=None, last=None):
    return orc.decode(case["q"], case["k"], case["v"],
                      case["indptr"] if indptr is None else indptr,
                      case["indices"] if indices is None else indices,
                      case["last"] if last is None else last,
                      dtype=case["dtype"], sm_scale=case["sm_scale"], rows=rows)


def dense_tokens(case, b, which):
    """[L, Hkv, D] float64 keys or values of request b, in sequence order."""
    pages = case["indices"][case["indptr"][b]:case["indptr"][b + 1]]
    pool = case[which + "64"]
    if len(pages) == 0:
        return np.zeros((0, case["hkv"], case["d"]))
    stacked = pool[pages].reshape(-1, case["hkv"], case["d"])
    return stacked[: case["lengths"][b]]


def check_bruteforce(orc):
    """Oracle vs torch SDPA + scipy logsumexp on dense gathered copies."""
    rng = np.random.default_rng(7)
    shapes = [(4, 2, 8, 1, "f16"), (4, 1, 8, 2, "bf16"), (2, 2, 4, 3, "f16"),
              (3, 3, 8, 2, "bf16"), (8, 2, 16, 4, "f16")]
    for hq, hkv, d, p, dtype in shapes:
        lengths = list(rng.integers(1, 3 * p + 3, size=3))
        case = paged_case(rng, lengths, hq, hkv, d, p, dtype)
        out, lse = run_case(orc, case)
        out = out.reshape(len(lengths), hq, d)
        lse = lse.reshape(len(lengths), hq)
        g = hq // hkv
        for b in range(len(lengths)):
            kd = torch.from_numpy(dense_tokens(case, b, "k"))      # [L, Hkv, D]
            vd = torch.from_numpy(dense_tokens(case, b, "v"))
            kq = kd.repeat_interleave(g, dim=1).permute(1, 0, 2)    # [Hq, L, D]
            vq = vd.repeat_interleave(g, dim=1).permute(1, 0, 2)
            qb = torch.from_numpy(case["q64"][b])                  # [Hq, D]
            ref = F.scaled_dot_product_attention(
                qb[None, :, None, :], kq[None], vq[None],
                scale=case["sm_scale"])[0, :, 0, :].numpy()
            logits = np.einsum("hd,hld->hl", case["q64"][b], kq.numpy()) \
                * case["sm_scale"]
            ref_lse = scipy.special.logsumexp(logits, axis=1)
            assert np.max(np.abs(out[b] - ref)) <= 1e-12, "bruteforce out"
            assert np.max(np.abs(lse[b] - ref_lse)) <= 1e-12, "bruteforce lse"


def check_single_key(orc):
    """n = 1: out is exactly v_0 and lse exactly sm_scale * <q, k_0>."""
    rng = np.random.default_rng(11)
    for dtype in ("f16", "bf16"):
        case = paged_case(rng, [1], 4, 2, 16, 4, dtype)
        # small integers: products and sums are exact in double
        for name in ("q", "k"):
            ints = rng.integers(-8, 9, size=case[name + "64"].shape).astype(np.float32)
            case[name], case[name + "64"] = _codes_and_values(ints, dtype)
        out, lse = run_case(orc, case)
        page, kvh = case["indices"][0], np.arange(4) // 2
        for h in range(4):
            k0 = case["k64"][page, 0, kvh[h]]
            v0 = case["v64"][page, 0, kvh[h]]
            assert np.array_equal(out[h], v0), "single key: out != v_0"
            dot = float(np.dot(case["q64"][0, h], k0))
            assert lse[h] == case["sm_scale"] * dot, "single key: lse != s_0"


def check_identical_keys(orc):
    """All keys equal: out = mean of V, lse = s + ln n."""
    rng = np.random.default_rng(12)
    for n, p in ((5, 2), (37, 8), (64, 16)):
        case = paged_case(rng, [n], 2, 1, 32, p, "f16")
        key = case["k64"][case["indices"][0], 0, 0].copy()
        codes, vals = _codes_and_values(
            np.broadcast_to(key.astype(np.float32), case["k64"].shape).copy(), "f16")
        case["k"], case["k64"] = codes, vals
        out, lse = run_case(orc, case)
        vd = dense_tokens(case, 0, "v")[:, 0, :]
        for h in range(2):
            s = case["sm_scale"] * math.fsum(case["q64"][0, h] * key)
            assert np.max(np.abs(out[h] - vd.mean(axis=0))) <= 1e-13, "identical keys out"
            assert abs(lse[h] - (s + math.log(n))) <= 1e-12, "identical keys lse"


def check_gqa_mapping(orc):
    """Query head h reads kv head h // g: kv head j holds values j + 1."""
    rng = np.random.default_rng(13)
    case = paged_case(rng, [9], 8, 4, 8, 4, "f16")
    vals = np.zeros(case["v64"].shape, dtype=np.float32)
    for j in range(4):
        vals[:, :, j, :] = j + 1
    case["v"], case["v64"] = _codes_and_values(vals, "f16")
    out, _ = run_case(orc, case)
    for h in range(8):
        assert np.max(np.abs(out[h] - (h // 2 + 1))) <= 1e-13, \
            "query head %d mapped wrongly" % h


def _sub_table(case, b, page_positions):
    """Table of request b restricted to the listed page positions."""
    pages = case["indices"][case["indptr"][b]:case["indptr"][b + 1]]
    npages = len(pages)
    chosen = sorted(page_positions, key=lambda i: (i == npages - 1, i))
    last = case["p"]
    if chosen and chosen[-1] == npages - 1:
        last = int(case["last"][b])
    indices = np.array([pages[i] for i in chosen], dtype=np.int32)
    return (np.array([0, len(chosen)], dtype=np.int32), indices,
            np.array([last if chosen else 0], dtype=np.int32))


def _state_of(orc, case, b, positions):
    indptr, indices, last = _sub_table(case, b, positions)
    return orc.decode(case["q"][b:b + 1], case["k"], case["v"], indptr,
                      indices, last, dtype=case["dtype"],
                      sm_scale=case["sm_scale"])


def check_union(orc):
    """merge(state(A), state(B)) = state(A u B) for disjoint page sets."""
    rng = np.random.default_rng(14)
    for dtype, p, n in (("f16", 4, 29), ("bf16", 1, 17), ("f16", 16, 100)):
        case = paged_case(rng, [n], 4, 2, 16, p, dtype)
        npages = (n + p - 1) // p
        full = list(range(npages))
        whole_out, whole_lse = _state_of(orc, case, 0, full)
        for _ in range(3):
            perm = list(rng.permutation(npages))
            cut1, cut2 = sorted(rng.integers(0, npages + 1, size=2))
            parts = [perm[:cut1], perm[cut1:cut2], perm[cut2:]]
            states = [_state_of(orc, case, 0, part) for part in parts]
            a, b, c = states
            left = orc.merge(*orc.merge(*a, *b), *c)
            right = orc.merge(*a, *orc.merge(*b, *c))
            for v, s in (left, right):
                assert np.max(np.abs(v - whole_out)) <= 1e-12, "union out"
                assert np.max(np.abs(s - whole_lse)) <= 1e-12, "union lse"


def check_empty(orc):
    """Empty rows give (0, -inf); an empty state is the merge identity."""
    rng = np.random.default_rng(15)
    case = paged_case(rng, [0, 7, 0], 4, 2, 8, 4, "f16")
    out, lse = run_case(orc, case)
    out = out.reshape(3, 4, 8)
    lse = lse.reshape(3, 4)
    for b in (0, 2):
        assert np.all(out[b] == 0.0) and np.all(lse[b] == -np.inf), "empty row"
    assert np.all(np.isfinite(lse[1])), "non-empty row"
    v, s = orc.merge(out[1], lse[1], out[0], lse[0])
    assert np.array_equal(v, out[1]) and np.array_equal(s, lse[1]), "identity (right)"
    v, s = orc.merge(out[0], lse[0], out[1], lse[1])
    assert np.array_equal(v, out[1]) and np.array_equal(s, lse[1]), "identity (left)"
    v, s = orc.merge(out[0], lse[0], out[2], lse[2])
    assert np.all(v == 0.0) and np.all(s == -np.inf), "empty u empty"


def check_permutation(orc):
    """Relabelling the pool's pages (and the page ids) changes nothing."""
    rng = np.random.default_rng(16)
    case = paged_case(rng, [13, 1, 24], 4, 2, 16, 4, "bf16", extra_pages=5)
    out, lse = run_case(orc, case)
    pool = case["k"].shape[0]
    pi = rng.permutation(pool)
    k2 = np.empty_like(case["k"])
    v2 = np.empty_like(case["v"])
    k2[pi] = case["k"]
    v2[pi] = case["v"]
    out2, lse2 = orc.decode(case["q"], k2, v2, case["indptr"],
                            pi[case["indices"]].astype(np.int32), case["last"],
                            dtype="bf16", sm_scale=case["sm_scale"])
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2), "permutation"


def check_extreme_shift(orc):
    """Every logit below -5e4: same output, lse shifted by the constant."""
    rng = np.random.default_rng(17)
    case = paged_case(rng, [23, 40], 4, 2, 16, 8, "f16")
    q32 = case["q64"].astype(np.float32)
    k32 = case["k64"].astype(np.float32)
    q32[..., 0] = 0.0
    base = dict(case)
    base["q"], base["q64"] = _codes_and_values(q32, "f16")
    out0, lse0 = run_case(orc, base)
    q32[..., 0] = 1024.0
    k32[..., 0] = -1024.0
    shifted = dict(case)
    shifted["q"], shifted["q64"] = _codes_and_values(q32, "f16")
    shifted["k"], shifted["k64"] = _codes_and_values(k32, "f16")
    out1, lse1 = run_case(orc, shifted)
    shift = -1024.0 * 1024.0 * case["sm_scale"]
    assert np.all(lse1 < -5e4), "logits not in the extreme range"
    assert np.all(np.isfinite(out1)), "non-finite output for extreme logits"
    assert np.max(np.abs(out1 - out0)) <= 1e-9, "extreme shift changed out"
    assert np.max(np.abs(lse1 - (lse0 + shift))) <= 1e-8, "extreme shift lse"


def check_wide_spread(orc):
    """Logits spread over thousands (exp would overflow without the max)."""
    rng = np.random.default_rng(18)
    case = paged_case(rng, [31, 6], 4, 2, 16, 4, "f16")
    q32 = case["q64"].astype(np.float32)
    k32 = case["k64"].astype(np.float32)
    q32[..., 0] = 256.0
    k32[..., 0] = rng.integers(-256, 257, size=k32.shape[:-1]).astype(np.float32)
    case["q"], case["q64"] = _codes_and_values(q32, "f16")
    case["k"], case["k64"] = _codes_and_values(k32, "f16")
    out, lse = run_case(orc, case)
    out = out.reshape(2, 4, 16)
    lse = lse.reshape(2, 4)
    for b in range(2):
        kq = torch.from_numpy(dense_tokens(case, b, "k")).repeat_interleave(
            2, dim=1).permute(1, 0, 2)
        vq = torch.from_numpy(dense_tokens(case, b, "v")).repeat_interleave(
            2, dim=1).permute(1, 0, 2)
        logits = np.einsum("hd,hld->hl", case["q64"][b], kq.numpy()) * case["sm_scale"]
        assert np.all(logits.max(axis=1) - logits.min(axis=1) > 1000.0)
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(case["q64"][b])[None, :, None, :], kq[None], vq[None],
            scale=case["sm_scale"])[0, :, 0, :].numpy()
        assert np.max(np.abs(out[b] - ref)) <= 1e-12, "wide spread out"
        assert np.max(np.abs(lse[b] - scipy.special.logsumexp(logits, axis=1))) \
            <= 1e-9, "wide spread lse"


def check_hnd_layout(orc):
    """HND copies of NHD pools (per page: heads before slots) give the same
    states, bit for bit; an NHD pool read as HND does not."""
    rng = np.random.default_rng(19)
    for p in (1, 3, 8):
        case = paged_case(rng, [2 * p + 1, 5 * p, 1], 8, 4, 16, p, "bf16")
        out, lse = run_case(orc, case)
        k_hnd = np.ascontiguousarray(case["k"].transpose(0, 2, 1, 3))
        v_hnd = np.ascontiguousarray(case["v"].transpose(0, 2, 1, 3))
        out2, lse2 = orc.decode(case["q"], k_hnd, v_hnd, case["indptr"],
                                case["indices"], case["last"], dtype="bf16",
                                sm_scale=case["sm_scale"], layout="HND")
        assert np.array_equal(out, out2) and np.array_equal(lse, lse2), "HND copy"
        if p > 1:
            out3, _ = orc.decode(case["q"], case["k"].reshape(k_hnd.shape),
                                 case["v"].reshape(v_hnd.shape), case["indptr"],
                                 case["indices"], case["last"], dtype="bf16",
                                 sm_scale=case["sm_scale"], layout="HND")
            assert not np.allclose(out, out3), "layout flag ignored"


ALL_CHECKS = [check_bruteforce, check_wide_spread, check_hnd_layout, check_single_key, check_identical_keys,
              check_gqa_mapping, check_union, check_empty, check_permutation,
              check_extreme_shift]


def failing_checks(orc):
    """Names of the checks this oracle fails (an exception counts)."""
    failed = []
    for check in ALL_CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(orc)
        except Exception:  # noqa: BLE001 - any failure is a detection
            failed.append(check.__name__)
    return failed
