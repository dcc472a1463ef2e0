"""Pins of the HFP4G32 oracle against what the HFP4 page and the mathematics fix.

Source: "HFP4" (hipfire.dev quant-formats), sections "Element format (OCP
E2M1)", "Block scale - UE8M0", "Per-row second-level scale (FP16)", "Byte
layout - HFP4G32", "Nibble packing", "Quantization recipe (HFP4G32)" and
"Validation".  The E2M1 tie rounding (ties to the even mantissa) is a stated
reading: the page does not fix it, so those cases are checked for validity
(both neighbours are equally near) rather than pinned.
"""
import math

import numpy as np
import pytest

import oracle
from synth import child_rngs, float32_to_bf16_bits, hfp4_gemv, normal_weights
from _helpers import bf16_bits_to_f64, decode_hfp4_independent, load_golden, rel_err_rows


def _mags():
    return np.array([oracle.e2m1_value(c) for c in range(8)])


def test_e2m1_lattice_facts_from_the_page():
    g = load_golden("hfp4_error_bound.txt")
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert len(vals) == g["e2m1_codes"]
    mags = sorted(set(abs(v) for v in vals))
    assert len(mags) == g["e2m1_magnitudes"]
    assert max(mags) == g["e2m1_max"] and min(vals) == -g["e2m1_max"]
    gaps = np.diff(mags)
    assert sorted(set(gaps)) == g["e2m1_gaps"]
    assert gaps.max() / 2 == g["largest_half_gap"]
    # code bit 3 is the sign; codes 0..7 are increasing magnitudes
    for c in range(8):
        assert oracle.e2m1_value(c | 8) == -oracle.e2m1_value(c) or c == 0
    assert list(_mags()) == sorted(_mags())


def test_e2m1_encode_is_nearest_on_a_dense_grid():
    mags = _mags()
    for v in np.linspace(-6.5, 6.5, 4001):
        c = oracle.e2m1_encode(v)
        err = abs(abs(v) - mags[c & 7])
        assert err <= np.min(np.abs(abs(v) - mags)) + 0.0
        assert (c >> 3) == (1 if math.copysign(1.0, v) < 0 else 0)
    # midpoints: both neighbours are equally near; the reading picks the even index
    for lo, hi in zip(range(7), range(1, 8)):
        mid = (mags[lo] + mags[hi]) / 2
        c = oracle.e2m1_encode(mid)
        assert c in (lo, hi) and c % 2 == 0


def test_ue8m0_matches_independent_decoder():
    import torch
    b = torch.arange(256, dtype=torch.uint8)
    try:
        ref = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    except Exception:
        pytest.skip("torch float8_e8m0fnu conversion unavailable")
    for e in range(255):
        assert oracle.ue8m0(e) == ref[e]
    assert math.isnan(oracle.ue8m0(255)) and math.isnan(ref[255])


def test_f16_rounding_matches_numpy():
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 1e-5, 500),
                         rng.normal(0, 1e4, 500)]).astype(np.float32)
    for x in xs:
        assert oracle.f32_to_f16_bits(x) == int(np.float16(x).view(np.uint16))
        assert oracle.f16_bits_to_f32(oracle.f32_to_f16_bits(x)) == np.float32(np.float16(x))


@pytest.mark.parametrize("K", [32, 256, 8192])
def test_row_sizes_and_header(K):
    g = load_golden("format_sizes.txt")
    M = 3
    assert oracle.hfp4_row_bytes(K) == g["hfp4_header_bytes"] + g["hfp4_block_bytes"] * K // 32
    bpw = oracle.hfp4_row_bytes(K) * 8 / K
    assert abs(bpw - (g["hfp4_payload_bpw"] + g["hfp4_header_bits_per_row"] / K)) < 1e-12
    W = hfp4_gemv(M=M, K=K)["W"]
    P = oracle.hfp4_pack(W)
    assert P.shape == (M, oracle.hfp4_row_bytes(K))
    for m in range(M):
        rs_bits = int(P[m, 0]) | (int(P[m, 1]) << 8)
        assert rs_bits == int(np.float16(np.abs(W[m]).max() / np.float32(6)).view(np.uint16))
        assert P[m, 2] == 0 and P[m, 3] == 0               # row_scale_b reserved = 0
        assert int(P[m, 4]) | (int(P[m, 5]) << 8) == K // 32
        assert P[m, 6] == 0                                 # no rotation flags
        assert not P[m, 7:16].any()                         # reserved bytes


def test_nibble_order_low_is_even():
    # max 6 -> row scale exactly 1.0; block max 6 -> e = 127; codes are exact
    w = np.zeros((1, 32), np.float32)
    w[0, 0], w[0, 1] = 6.0, -0.5      # codes 7 and 9
    w[0, 2], w[0, 3] = 1.5, -4.0      # codes 3 and 14
    P = oracle.hfp4_pack(w)
    assert P[0, 16] == 127
    assert P[0, 17] == 0x97
    assert P[0, 18] == 0xE3
    dec = oracle.hfp4_decode(P, 1, 32)
    np.testing.assert_array_equal(dec[0, :4], [6.0, -0.5, 1.5, -4.0])


def test_block_exponent_is_smallest_covering():
    W = hfp4_gemv(M=16, K=512)["W"]
    W[3, 64:96] *= 1e-3   # a quiet block
    W[5, :32] = 0.0       # an all-zero block
    P = oracle.hfp4_pack(W)
    for m in range(16):
        rs = float(np.float16(np.abs(W[m]).max() / np.float32(6)))
        for j in range(16):
            e = int(P[m, 16 + 17 * j])
            bmax = float(np.abs(W[m, 32 * j:32 * j + 32] / np.float32(rs)).max())
            assert bmax <= 6.0 * 2.0 ** (e - 127)
            if e > 0:
                assert bmax > 6.0 * 2.0 ** (e - 128)
    assert P[5, 16] == 0


@pytest.mark.parametrize("scale", [0.02, 1.0, 3e-3, 50.0])
def test_round_trip_error_bound(scale):
    rng = np.random.default_rng(17)
    M, K = 12, 1024
    W = (rng.standard_t(4, (M, K)) * scale).astype(np.float32)
    P = oracle.hfp4_pack(W)
    D = oracle.hfp4_decode(P, M, K)
    mags = _mags()
    half_gaps = np.diff(mags) / 2
    for m in range(M):
        rs = float(np.float16(np.abs(W[m]).max() / np.float32(6)))
        for j in range(K // 32):
            e = int(P[m, 16 + 17 * j])
            unit = rs * 2.0 ** (e - 127)
            err = np.abs(W[m, 32 * j:32 * j + 32].astype(np.float64) - D[m, 32 * j:32 * j + 32])
            # global bound of the page (+ the fp32 rounding of W / row_scale_a)
            slack = np.abs(W[m, 32 * j:32 * j + 32]) * 2.0 ** -23
            assert np.all(err <= unit * 1.0 + slack)
            # local half-gap: the error never exceeds half the gap it falls in
            v = np.abs(W[m, 32 * j:32 * j + 32].astype(np.float64)) / unit
            idx = np.clip(np.searchsorted(mags, v) - 1, 0, 6)
            assert np.all(err <= unit * half_gaps[idx] + slack + 1e-300)


def test_zero_row_and_rejections():
    W = np.zeros((2, 64), np.float32)
    W[1] = 1.0
    P = oracle.hfp4_pack(W)
    assert not P[0, :2].any() and not P[0, 16:].any()
    np.testing.assert_array_equal(oracle.hfp4_decode(P, 2, 64)[0], 0.0)
    with pytest.raises(ValueError):
        oracle.hfp4_pack(np.zeros((1, 40), np.float32))
    big = np.full((1, 32), 1e6, np.float32)   # 1e6/6 overflows fp16
    with pytest.raises(ValueError):
        oracle.hfp4_pack(big)


def test_block_nan_byte_decodes_to_nan():
    P = oracle.hfp4_pack(hfp4_gemv(M=1, K=64)["W"])
    P[0, 16 + 17] = 0xFF
    D = oracle.hfp4_decode(P, 1, 64)
    assert np.all(np.isnan(D[0, 32:])) and not np.any(np.isnan(D[0, :32]))


def test_gemv_loop_formula_matches_decoded_dot():
    w = hfp4_gemv(M=40, K=1024, N=3)
    P = oracle.hfp4_pack(w["W"])
    y = oracle.hfp4_gemv(P, 40, 1024, w["x"])
    ref = w["x"].astype(np.float64) @ oracle.hfp4_decode(P, 40, 1024).T
    assert np.all(rel_err_rows(y, ref) <= 1e-12)
    rows = np.array([39, 2])
    np.testing.assert_array_equal(oracle.hfp4_gemv(P, 40, 1024, w["x"], rows=rows), y[:, rows])
    # decoded weights approximate W within the format's error (sanity, not a pin)
    assert np.all(rel_err_rows(ref, w["x"].astype(np.float64) @ w["W"].T.astype(np.float64)) < 0.2)


def test_decode_matches_independent_decoder():
    w = hfp4_gemv(M=24, K=512, N=1)
    P = oracle.hfp4_pack(w["W"])
    P[3, 16 + 17 * 2] = 0xFF   # a NaN block
    P[5, 16] = 0x00            # the subnormal block scale 2^-127
    np.testing.assert_array_equal(oracle.hfp4_decode(P, 24, 512), decode_hfp4_independent(P, 24, 512))


def test_gemm_matches_independent_decoded_product():
    """Prefill: Y = X W^T over bf16 tokens (no activation quantization), against
    numpy's product of the independently decoded weights in fp64."""
    r_w, r_x = child_rngs(21, 2)
    M, K, N = 36, 768, 5
    P = oracle.hfp4_pack(normal_weights(r_w, M, K, 0.03))
    X = float32_to_bf16_bits(r_x.standard_normal((N, K)).astype(np.float32))
    Y = oracle.hfp4_gemm(P, M, K, X)
    ref = bf16_bits_to_f64(X) @ decode_hfp4_independent(P, M, K).T
    assert np.all(rel_err_rows(Y, ref) <= 1e-12)
    rows = np.array([35, 0, 17])
    np.testing.assert_array_equal(oracle.hfp4_gemm(P, M, K, X, rows=rows), Y[:, rows])


def test_gemm_exact_when_every_weight_is_on_the_lattice():
    """Rows holding 6 have row_scale_a = 1 and every value of {+-6, +-3, +-1.5,
    +-1, 0} on its block lattice, so the packing is exact and, with small
    integer tokens, so is every output."""
    rng = np.random.default_rng(5)
    M, K, N = 8, 256, 3
    W = rng.choice(np.array([-6.0, -3.0, -1.5, -1.0, 0.0, 1.0, 1.5, 3.0, 6.0]), (M, K))
    W[:, 0] = 6.0
    P = oracle.hfp4_pack(W.astype(np.float32))
    np.testing.assert_array_equal(oracle.hfp4_decode(P, M, K), W)
    Xf = rng.integers(-8, 9, (N, K)).astype(np.float32)
    Y = oracle.hfp4_gemm(P, M, K, float32_to_bf16_bits(Xf))
    np.testing.assert_array_equal(Y, Xf.astype(np.float64) @ W.T)
