"""The exact near-half rounding rule of the decode GEMV's in-kernel quantize,
checked on the CPU against IEEE float32 division.

The kernel computes q = roundf(fl(a / d)) (the Q8_1 quantizer of the
"ROCmFP2 codebook research report", 03 Runtime: d = amax / 127, q =
round(a / d)) from z = a * rcp.approx(d).  For the rare values whose z lies
within 2^-12 of a half-integer it does not divide: with A = |a| and H =
floor(|z|) + 1/2, fl(A/d) >= H exactly when A - H*d >= -(u/2)*d, u being the
float spacing just below H.  This file re-derives that rule in numpy, with
float32 rounding emulated exactly through float64, and checks

- that the two products it relies on, R = A - H*d and (u/2)*d, are exact in
  float32 (the FMA residual and a power-of-two scaling), and
- that the decision equals roundf of numpy's correctly rounded float32
  quotient for every half-integer H = 0.5 .. 126.5, scales over 200 binades
  and numerators up to 64 ulps either side of H*d.

The kernel's own results are compared with the oracle, bit for bit, by the
"ties" and "near_half" kinds of tests/test_gpu_gemv.py.
"""
import numpy as np

F32 = np.float32


def rn32(v):
    """Round float64 values to the nearest float32 (ties to even)."""
    return np.asarray(v, np.float64).astype(F32)


def half_spacing_below(H):
    """u/2 for float32 H > 0: half the distance from H to the next float below."""
    bits = np.asarray(H, F32).view(np.uint32)
    drop = np.where((bits & 0x7FFFFF) == 0, 25, 24).astype(np.uint32)
    return (((bits >> 23) - drop) << 23).view(F32)


def decide(a, d, H):
    """The kernel's rule: roundf(fl(a/d)) for a/d near +-H."""
    A = np.abs(a).astype(np.float64)
    R = rn32(A - H.astype(np.float64) * d.astype(np.float64))  # fmaf(-H, d, A)
    t = rn32(half_spacing_below(H).astype(np.float64) * d.astype(np.float64))
    up = (R > -t) | ((R == -t) & ((H.view(np.uint32) & 1) == 0))
    return np.copysign((H - F32(0.5)) + np.where(up, F32(1), F32(0)), a).astype(F32)


def reference(a, d):
    """roundf of the IEEE float32 quotient (halves away from zero)."""
    q = (a / d).astype(F32)
    return (np.sign(q) * np.floor(np.abs(q).astype(np.float64) + 0.5)).astype(F32)


def cases(rng, n_d=64, ulps=64):
    """Numerators within `ulps` float steps of H*d for every H and random d."""
    H = (np.arange(127, dtype=F32) + F32(0.5))                       # 0.5 .. 126.5
    e = rng.integers(-100, 100, n_d)
    d = (rng.uniform(1.0, 2.0, n_d) * np.exp2(e)).astype(F32)
    d = np.concatenate([d, F32([1.0, 2.0 ** -100, 1.0 / 127, 3.0 ** 5])]).astype(F32)
    center = rn32(H[:, None].astype(np.float64) * d[None, :].astype(np.float64))
    k = np.arange(-ulps, ulps + 1)
    bits = center.view(np.int32)[..., None] + k                       # neighbours of H*d
    a = bits.astype(np.int32).view(F32)
    Hs = np.broadcast_to(H[:, None, None], a.shape)
    ds = np.broadcast_to(d[None, :, None], a.shape)
    sign = np.where(rng.random(a.shape) < 0.5, F32(-1), F32(1))
    return (a * sign).ravel(), ds.ravel().astype(F32), Hs.ravel().astype(F32)


def test_products_are_exact():
    a, d, H = cases(np.random.default_rng(1))
    A = np.abs(a).astype(np.float64)
    exact_R = A - H.astype(np.float64) * d.astype(np.float64)
    assert np.array_equal(rn32(exact_R).astype(np.float64), exact_R)
    exact_t = half_spacing_below(H).astype(np.float64) * d.astype(np.float64)
    assert np.array_equal(rn32(exact_t).astype(np.float64), exact_t)


def test_half_spacing_below():
    H = (np.arange(127, dtype=F32) + F32(0.5))
    below = (H.view(np.uint32) - 1).view(F32)                          # the float just below H
    assert np.array_equal(half_spacing_below(H), ((H - below) / 2).astype(F32))


def test_rule_matches_ieee_division():
    for seed in range(4):
        a, d, H = cases(np.random.default_rng(10 + seed))
        near = np.abs(np.abs(a.astype(np.float64) / d) - H) < 2.0 ** -12 + 2.0 ** -14
        assert near.mean() > 0.5  # the neighbourhood the kernel hands to the rule
        np.testing.assert_array_equal(decide(a[near], d[near], H[near]), reference(a[near], d[near]))


def test_rule_sees_both_outcomes_and_exact_halves():
    a, d, H = cases(np.random.default_rng(7), n_d=8, ulps=4)
    ref = reference(a, d)
    got = decide(a, d, H)
    np.testing.assert_array_equal(got, ref)
    mag = np.abs(ref) - (H - F32(0.5))
    assert set(np.unique(mag).tolist()) == {0.0, 1.0}  # toward and away from zero both occur
    exact = (np.abs(a).astype(np.float64) == H.astype(np.float64) * d.astype(np.float64))
    assert exact.any() and np.all(mag[exact] == 1.0)   # an exact half goes away from zero
