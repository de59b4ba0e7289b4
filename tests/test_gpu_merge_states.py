"""GPU merge_states against the oracle merge ("FlashInfer"
(aiwiki.ai/wiki/flashinfer), "Attention states"; -inf handling from
"Extreme-negative-logit correction")."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_plan_gb300 as pkd
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def random_states(rng, n, h, d, dtype, empty_frac=0.2):
    v = torch.from_numpy(rng.standard_normal((n, h, d)).astype(np.float32)).to(
        DTYPES[dtype])
    s = (rng.standard_normal((n, h)) * 20).astype(np.float32)
    s[rng.random((n, h)) < empty_frac] = -np.inf
    v_np = v.float().numpy()
    v_np[np.isneginf(s)] = 0.0
    v = torch.from_numpy(v_np).to(DTYPES[dtype])
    return v, torch.from_numpy(s)


def check(v, s, v_ref, s_ref, dtype):
    """The decode tests' bounds: |dv| <= 5e-3 where |ref| < 2, plus the output
    type's half-ulp where |ref| >= 2 (fp32 outputs are held to 1e-5
    everywhere); |ds| <= 1e-3 + 2 ulp_fp32(|s|); two empty sides give exactly
    (0, -inf)."""
    v = v.float().cpu().numpy().astype(np.float64).reshape(v_ref.shape)
    s = s.cpu().numpy().astype(np.float64).reshape(s_ref.shape)
    both_empty = np.isneginf(s_ref)
    assert np.all(np.isneginf(s[both_empty])) and np.all(v[both_empty] == 0)
    assert np.all(np.isfinite(v))
    err = np.abs(v - v_ref)
    if dtype == "f32":
        bound = np.full_like(err, 1e-5)
    else:
        large = np.abs(v_ref) >= 2.0
        bound = gh.OUT_TOL + np.where(large, gh.half_ulp(v_ref, dtype), 0.0)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert np.all(err <= bound), "v error %.3g at %s (ref %.4g)" % (
        err[worst], worst, v_ref[worst])
    fin = ~both_empty
    if fin.any():
        s_err = np.abs(s[fin] - s_ref[fin])
        s_bound = gh.LSE_TOL + 2.0 * np.spacing(
            np.abs(s_ref[fin]).astype(np.float32)).astype(np.float64)
        assert np.all(s_err <= s_bound), "s error %.3g" % s_err.max()


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("n,h,d", [(1, 1, 8), (37, 32, 128), (128, 32, 128), (5, 3, 1024)])
def test_merge_states_matches_oracle(dtype, n, h, d):
    rng = np.random.default_rng(n * 1000 + h + d)
    va, sa = random_states(rng, n, h, d, dtype)
    vb, sb = random_states(rng, n, h, d, dtype)
    out_v, out_s = pkd.merge_states(va.cuda(), sa.cuda(), vb.cuda(), sb.cuda())
    torch.cuda.synchronize()
    v_ref, s_ref = oracle.merge(va.double().numpy(), sa.double().numpy(),
                                vb.double().numpy(), sb.double().numpy())
    check(out_v, out_s, v_ref, s_ref, dtype)


def test_merge_states_in_place_and_associative():
    rng = np.random.default_rng(3)
    n, h, d = 64, 8, 128
    states = [random_states(rng, n, h, d, "f32", 0.1) for _ in range(3)]
    dev = [(v.cuda(), s.cuda()) for v, s in states]
    (va, sa), (vb, sb), (vc, sc) = dev
    left = pkd.merge_states(*pkd.merge_states(va, sa, vb, sb), vc, sc)
    bc = pkd.merge_states(vb, sb, vc, sc)
    right = pkd.merge_states(va, sa, *bc)
    torch.cuda.synchronize()
    assert torch.allclose(left[0], right[0], atol=1e-5)
    assert torch.allclose(left[1], right[1], atol=1e-4, equal_nan=False)
    # in place: the output overwrites side a
    va2, sa2 = va.clone(), sa.clone()
    pkd.merge_states(va2, sa2, vb, sb, v_out=va2, s_out=sa2)
    ref = pkd.merge_states(va, sa, vb, sb)
    torch.cuda.synchronize()
    assert torch.equal(va2, ref[0]) and torch.equal(sa2, ref[1])


def test_merge_states_identity_and_both_empty():
    n, h, d = 4, 2, 16
    v = torch.randn(n, h, d, device="cuda", dtype=torch.float16)
    s = torch.randn(n, h, device="cuda") * 5
    empty_v = torch.zeros_like(v)
    empty_s = torch.full_like(s, -float("inf"))
    mv, ms = pkd.merge_states(v, s, empty_v, empty_s)
    torch.cuda.synchronize()
    assert torch.equal(mv, v) and torch.equal(ms, s)
    mv, ms = pkd.merge_states(empty_v, empty_s, empty_v, empty_s)
    torch.cuda.synchronize()
    assert torch.all(mv == 0) and torch.all(torch.isneginf(ms))


def test_merge_states_rejects_bad_shapes():
    v = torch.zeros(2, 2, 12, device="cuda")
    s = torch.zeros(2, 2, device="cuda")
    with pytest.raises(pkd.PkdError) as e:
        pkd.merge_states(v, s, v, s)
    assert e.value.status == -4


@pytest.mark.parametrize("seed", range(12))
def test_merge_states_random_shapes(seed):
    """Seeded draws of n (0 included), heads, head_dim (multiples of 8 up to
    1024), dtype, the share of empty states and the spread of s, each against
    the oracle merge."""
    rng = np.random.default_rng([9001, seed])
    n = int(rng.choice([0, 1, 2, 7, 65, 300]))
    h = int(rng.integers(1, 65))
    d = 8 * int(rng.integers(1, 129))
    dtype = ["f16", "bf16", "f32"][seed % 3]
    empty = float(rng.choice([0.0, 0.1, 0.5, 1.0]))
    va, sa = random_states(rng, n, h, d, dtype, empty)
    vb, sb = random_states(rng, n, h, d, dtype, empty)
    spread = float(rng.choice([1.0, 100.0, 1e4]))
    sa = sa * spread / 20
    sb = sb * spread / 20
    out_v, out_s = pkd.merge_states(va.cuda(), sa.cuda(), vb.cuda(), sb.cuda())
    torch.cuda.synchronize()
    if n == 0:
        assert out_v.numel() == 0 and out_s.numel() == 0
        return
    v_ref, s_ref = oracle.merge(va.double().numpy(), sa.double().numpy(),
                                vb.double().numpy(), sb.double().numpy())
    check(out_v, out_s, v_ref, s_ref, dtype)
