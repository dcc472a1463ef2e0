"""Pins of the oracle's block-scaled FP4 (NVFP4) functions.

Each test checks the oracle against something it does not share code with:
torch's own float8_e4m3fn cast and decode, the E2M1 lattice of the "HFP4"
page ("Element format (OCP E2M1)"), the exact ROCmFP2 decode ("ROCmFP2
codebook research report", "02 Quantization"), a hand-derived block
(tests/golden/nvfp4_act_example.txt), closed forms and the rounding bound.
"""
import os

import numpy as np
import pytest

import oracle
from synth import child_rngs, normal_weights

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_act_example.txt")
# "HFP4" page, "Element format (OCP E2M1)": magnitudes of codes 0..7; bit 3 is the sign.
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1(codes):
    codes = np.asarray(codes).astype(np.int64)
    v = E2M1_MAG[codes & 7]
    return np.where(codes & 8, -v, v)


def torch_e4m3(b):
    t = torch.tensor(np.asarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3_encode(v):
    return torch.tensor(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3fn_decode_matches_torch():
    ours = np.array([oracle.e4m3fn_value(b) for b in range(256)])
    ref = torch_e4m3(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan[0x7F] and nan[0xFF]
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3fn_encode_matches_torch():
    rng = np.random.default_rng(5)
    grid = torch_e4m3(np.arange(0x7F))
    mids = (grid[:-1] + grid[1:]) / 2  # exact ties
    v = np.concatenate([rng.uniform(0, 448, 3000), np.exp(rng.uniform(-9, 6, 3000)), mids, grid,
                        [0.0, 2.0 ** -10, 448.0]]).astype(np.float32)
    v = v[v <= 448]
    ours = np.array([oracle.e4m3fn_encode(float(t)) for t in v])
    assert np.array_equal(ours, torch_e4m3_encode(v))
    # above the largest finite value the encoder saturates at 448 (0x7E)
    assert oracle.e4m3fn_encode(449.0) == 0x7E and oracle.e4m3fn_encode(1e6) == 0x7E


def test_rfp2_weights_are_exact_nvfp4():
    """codebook * s(b) == E2M1 * E4M3FN(b) for every code and legal byte, and
    the converted blocks dequantize (torch's E4M3FN, the page's E2M1 lattice)
    to exactly the ROCmFP2 weights."""
    K = 32 * 127
    rng = np.random.default_rng(9)
    blocks = np.zeros((1, K // 32, 10), np.uint8)
    blocks[0, :, :8] = rng.integers(0, 256, (K // 32, 8), dtype=np.uint8)
    blocks[0, :, 8] = np.arange(127)  # every legal scale byte
    blocks[0, :, 9] = np.arange(127)[::-1]
    for P, M in [(blocks.reshape(1, -1), 1),
                 (oracle.rfp2_pack(normal_weights(child_rngs(4, 1)[0], 8, 512, 0.02)), 8)]:
        Kp = P.size // M // 10 * 32
        codes, sb = oracle.rfp2_to_nvfp4(P, M, Kp)
        assert set(np.unique(codes & 7).tolist()) <= {1, 4}  # only +-0.5 and +-2
        val = e2m1(codes) * np.repeat(torch_e4m3(sb), 16, axis=1)
        assert np.array_equal(val, oracle.rfp2_decode(P, M, Kp).astype(np.float64))


def test_nvfp4_act_golden():
    rows = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, *vals = line.split()
            rows[k] = vals
    x = np.array([float(v) for v in rows["x"]], np.float32)[None]
    codes, sb, g = oracle.nvfp4_quant_act(x)
    assert g[0] == float(rows["g"][0])
    assert sb[0, 0] == int(rows["scale_byte"][0], 16)
    assert codes[0].tolist() == [int(v) for v in rows["codes"]]


def _rows(kind, rng, N, K):
    if kind == "normal":
        return rng.standard_normal((N, K)).astype(np.float32)
    if kind == "heavy":
        return (rng.standard_t(2, (N, K)) * 3).astype(np.float32)
    if kind == "sparse":
        x = rng.standard_normal((N, K)).astype(np.float32)
        x[rng.random((N, K)) < 0.7] = 0.0
        x[0, :32] = 0.0  # whole zero blocks
        return x
    if kind == "tiny":
        return (rng.standard_normal((N, K)) * 1e-30).astype(np.float32)
    if kind == "wide":  # blocks far below the row maximum: small scale bytes, subnormal ones
        x = rng.standard_normal((N, K)).astype(np.float32)
        x *= np.float32(2.0) ** rng.integers(-40, 1, (N, K // 16)).repeat(16, axis=1).astype(np.float32)
        return x
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "heavy", "sparse", "tiny", "wide"])
def test_nvfp4_act_properties(kind):
    """Scale bytes are torch's rounding of (bmax/6)*g; each code is a nearest
    lattice point of x*g/s (ties to the even index); the value is within
    s/g of x; the row maximum maps to +-6 at scale 448; zero blocks store +0."""
    rng = np.random.default_rng(len(kind))
    N, K = 3, 512
    x = _rows(kind, rng, N, K)
    codes, sb, g = oracle.nvfp4_quant_act(x)
    f32 = np.float32
    amax = np.abs(x).max(axis=1)
    assert np.array_equal(g, np.where(amax > 0, f32(2688) / np.where(amax > 0, amax, 1), f32(1)))
    bmax = np.abs(x).reshape(N, K // 16, 16).max(axis=2)
    t = (bmax / f32(6)) * g[:, None]
    assert np.array_equal(sb, torch_e4m3_encode(np.minimum(t, f32(448))))
    s = torch_e4m3(sb)
    sk = np.repeat(s, 16, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = ((x * g[:, None]) / np.repeat(s.astype(np.float32), 16, axis=1)).astype(np.float64)
    e[sk == 0] = 0.0
    dist = np.abs(np.abs(e)[..., None] - E2M1_MAG)  # distance to every magnitude
    best = dist.min(axis=-1)
    mag = codes & 7
    assert np.array_equal(dist[np.arange(N)[:, None], np.arange(K)[None], mag], best)
    tie = (dist == best[..., None]).sum(-1) > 1
    assert np.all(mag[tie] % 2 == 0)
    nz = (sk > 0) & (mag > 0)
    assert np.all(((codes & 8) > 0)[nz] == (x < 0)[nz])
    assert np.all(codes[sk == 0] == 0)
    # error bound: |e| <= 6 t / s, so the scaled error is at most the largest
    # half-gap (1) or the saturation excess 6 (t/s - 1); a block whose scale
    # byte is 0 stores 0, off by at most bmax = 6 t / g
    xhat = e2m1(codes) * sk / g[:, None].astype(np.float64)
    tk = np.repeat(t.astype(np.float64), 16, axis=1)
    gk = g[:, None].astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        bound = np.where(sk > 0, sk / gk * np.maximum(1.0, 6.0 * (tk / sk - 1.0)), 6.0 * tk / gk)
    assert np.all(np.abs(xhat - x) <= bound * (1 + 1e-6))
    for n in range(N):
        if amax[n] > 0:
            k = int(np.argmax(np.abs(x[n])))
            assert sb[n, k // 16] == 0x7E and (codes[n, k] & 7) == 7


def test_nvfp4_act_power_of_two_invariance():
    """Scaling a row by 2^j leaves every code and scale byte as it is and
    divides g by 2^j (all steps are exact under power-of-two scaling)."""
    x = np.random.default_rng(3).standard_normal((2, 256)).astype(np.float32)
    c0, s0, g0 = oracle.nvfp4_quant_act(x)
    for j in (-20, -3, 5, 30):
        c1, s1, g1 = oracle.nvfp4_quant_act(x * np.float32(2.0 ** j))
        assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
        assert np.array_equal(g1, g0 / np.float32(2.0 ** j))


def test_nvfp4_gemm_is_the_dequantized_dot():
    """The product is the fp64 dot of the dequantized operands (torch's
    E4M3FN, the page's lattice), divided by g only once."""
    rng = np.random.default_rng(11)
    M, K, N = 5, 256, 3
    P = oracle.rfp2_pack(normal_weights(child_rngs(7, 1)[0], M, K, 0.03))
    wc, ws = oracle.rfp2_to_nvfp4(P, M, K)
    x = rng.standard_normal((N, K)).astype(np.float32)
    xc, xs, g = oracle.nvfp4_quant_act(x)
    W = e2m1(wc) * np.repeat(torch_e4m3(ws), 16, axis=1)
    X = e2m1(xc) * np.repeat(torch_e4m3(xs), 16, axis=1) / g[:, None].astype(np.float64)
    ref = X @ W.T
    got = oracle.nvfp4_gemm(wc, ws, M, K, xc, xs, g)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # rows made of E2M1 values times a power of two per block, each block
    # holding a +-6 * 2^q and the row maximum 6 * 2^q0, are on their own NVFP4
    # grid (g = 448 * 2^-q0, scales 448 * 2^(q - q0), all exact), so the
    # product is the exact product with the ROCmFP2 weights
    q0 = 3
    qb = rng.integers(q0 - 8, q0 + 1, (N, K // 16))
    qb[:, 0] = q0
    cg = rng.integers(0, 16, (N, K))
    cg[:, ::16] = np.where(rng.random((N, K // 16)) < 0.5, 7, 15)
    xg = (e2m1(cg) * np.exp2(np.repeat(qb, 16, axis=1))).astype(np.float32)
    c2, s2, g2 = oracle.nvfp4_quant_act(xg)
    assert np.all(g2 == np.float32(448 * 2.0 ** -q0))
    X2 = e2m1(c2) * np.repeat(torch_e4m3(s2), 16, axis=1) / g2[:, None].astype(np.float64)
    np.testing.assert_array_equal(X2, xg.astype(np.float64))
    exact = xg.astype(np.float64) @ oracle.rfp2_decode(P, M, K).astype(np.float64).T
    np.testing.assert_allclose(oracle.nvfp4_gemm(wc, ws, M, K, c2, s2, g2), exact, rtol=1e-12, atol=0)
