"""Pins of the ROCmFP2 oracle against what the pages and the mathematics fix.

Sources: "ROCmFP2 codebook research report", sections "01 Storage",
"02 Quantization" and "03 Runtime".  No test here needs a GPU.
"""
import math

import numpy as np
import pytest

import oracle
from synth import decode_gemv, moe_gemv, normal_activations, tiny_gemv
from _helpers import (decode_weights_independent, e4m3fn_half_table, load_golden, rel_err_rows,
                      unpack_codes)


# -- worked example (02 Quantization) -----------------------------------------

def test_worked_example_codes_byte_and_reconstruction():
    g = load_golden("rfp2_worked_example.txt")
    s = oracle.ue4m3(g["scale_byte"])
    assert s == g["scale"]
    vals = np.array(g["values"], np.float32)
    codes = [oracle.rfp2_code(v, s) for v in vals]
    assert codes == [int(c) for c in g["codes"]]
    assert [oracle.codebook_value(c) for c in codes] == [int(v) for v in g["levels"]]
    # Pack a half whose values are exactly the example's reconstruction: the only
    # scale that reproduces +-0.5 and +-2 with the levels {1, 4} is 0.5, so the
    # search must pick 0x38 and the first code byte must be the page's 0xE4.
    recon = np.array(g["reconstruction"], np.float32)
    W = np.tile(recon, 8).reshape(1, 32)
    P = oracle.rfp2_pack(W)
    assert P.shape == (1, 1, 10)
    assert P[0, 0, 8] == g["scale_byte"] and P[0, 0, 9] == g["scale_byte"]
    assert all(P[0, 0, j] == g["packed_byte"] for j in range(8))
    dec = oracle.rfp2_decode(P, 1, 32)
    np.testing.assert_array_equal(dec[0, :4], recon)


def test_decode_of_page_byte():
    g = load_golden("rfp2_worked_example.txt")
    blk = np.zeros((1, 1, 10), np.uint8)
    blk[0, 0, 0] = g["packed_byte"]
    blk[0, 0, 8] = g["scale_byte"]
    blk[0, 0, 9] = g["scale_byte"]
    dec = oracle.rfp2_decode(blk, 1, 32)
    np.testing.assert_array_equal(dec[0, :4], np.array(g["reconstruction"], np.float32))
    # the other code bytes are 0 -> level -4 at scale 0.5
    np.testing.assert_array_equal(dec[0, 4:], np.full(28, -2.0, np.float32))


# -- UE4M3 scale byte ---------------------------------------------------------

def test_ue4m3_page_facts():
    g = load_golden("ue4m3_scale_byte.txt")
    legal = []
    for b in range(256):
        try:
            legal.append((b, oracle.ue4m3(b)))
        except ValueError:
            pass
    assert len(legal) == g["legal_count"]
    assert [b for b, _ in legal] == list(range(g["first_rejected"]))
    positives = [s for _, s in legal if s > 0]
    assert min(positives) == g["smallest_positive"]
    assert max(positives) == g["largest"]
    # strictly increasing: every legal byte names a distinct scale
    ss = [s for _, s in legal]
    assert all(a < b for a, b in zip(ss, ss[1:]))


def test_ue4m3_equals_half_of_e4m3fn_from_an_independent_decoder():
    """UE4M3(b) is half the OCP E4M3FN value of the same byte (torch's decoder)."""
    table = e4m3fn_half_table()
    for b in range(0x7F):
        assert oracle.ue4m3(b) == table[b], hex(b)
    assert math.isnan(table[0x7F])  # the byte the page rejects is E4M3FN's NaN


# -- code choice ----------------------------------------------------------------

def test_code_choice_boundaries():
    s = np.float32(0.5)
    at = np.float32(1.25)  # |x/s| == 2.5 exactly -> inner
    assert oracle.rfp2_code(at, s) == 2
    assert oracle.rfp2_code(-at, s) == 1
    above = np.nextafter(at, np.float32(10))
    assert oracle.rfp2_code(above, s) == 3
    assert oracle.rfp2_code(-above, s) == 0
    # zeros go to the positive inner level; s == 0 keeps inner levels by sign
    assert oracle.rfp2_code(0.0, s) == 2
    assert oracle.rfp2_code(-0.0, s) == 2
    assert oracle.rfp2_code(5.0, 0.0) == 2
    assert oracle.rfp2_code(-5.0, 0.0) == 1


# -- scale search: brute force with an independent implementation ---------------

def _independent_search(halves: np.ndarray):
    """numpy: for every half and every legal byte, codes and fp64 SSE summed in
    index order; first argmin wins."""
    table = e4m3fn_half_table()[:0x7F].astype(np.float32)        # [127]
    x = halves.astype(np.float32)[:, None, :]                      # [H, 1, 16]
    s = table[None, :, None]                                       # [1, 127, 1]
    with np.errstate(divide="ignore", invalid="ignore"):
        mag = np.abs(x / s)
    inner = np.where(s == 0, True, mag <= np.float32(2.5))
    neg = x < 0
    level = np.where(inner, 1.0, 4.0) * np.where(neg, -1.0, 1.0)
    recon = (level.astype(np.float32) * s) * np.where(s == 0, 0.0, 1.0)
    err = x.astype(np.float64) - recon.astype(np.float64)
    sse = np.zeros(err.shape[:2])
    for i in range(16):
        sse = sse + err[:, :, i] * err[:, :, i]
    best = np.argmin(sse, axis=1)
    return best, sse


@pytest.mark.parametrize("kind", ["normal", "student_t", "tiny", "huge", "sparse", "mixed"])
def test_scale_search_is_exhaustive_argmin(kind):
    rng = np.random.default_rng(123)
    H = 400
    if kind == "normal":
        halves = rng.normal(0, 0.02, (H, 16))
    elif kind == "student_t":
        halves = rng.standard_t(5, (H, 16)) * 0.02
    elif kind == "tiny":
        halves = rng.normal(0, 1e-4, (H, 16))
    elif kind == "huge":
        halves = rng.normal(0, 300.0, (H, 16))
    elif kind == "sparse":
        halves = rng.normal(0, 0.5, (H, 16)) * (rng.random((H, 16)) < 0.2)
    else:
        halves = rng.normal(0, 1, (H, 16)) * 10.0 ** rng.integers(-5, 3, (H, 1))
    halves = halves.astype(np.float32)
    best, sse = _independent_search(halves)
    for h in range(H):
        b, codes = oracle.rfp2_quantize_half(halves[h])
        assert b == best[h], (kind, h)
        assert oracle.rfp2_half_sse(halves[h], b) == sse[h, b]
        assert sse[h, b] <= sse[h].min()


def test_zero_half_picks_byte_zero():
    b, codes = oracle.rfp2_quantize_half(np.zeros(16, np.float32))
    assert b == 0 and np.all(codes == 2)
    b, codes = oracle.rfp2_quantize_half(-np.zeros(16, np.float32))
    assert b == 0 and np.all(codes == 2)


def test_exact_levels_are_reproduced_exactly():
    """Any half made of levels*s for a legal s has zero error at s."""
    table = e4m3fn_half_table()
    rng = np.random.default_rng(7)
    for b in range(1, 0x7F):
        s = np.float32(table[b])
        lv = rng.choice([-4.0, -1.0, 1.0, 4.0], 16).astype(np.float32)
        x = lv * s
        bb, codes = oracle.rfp2_quantize_half(x)
        assert oracle.rfp2_half_sse(x, bb) == 0.0
        rec = np.array([oracle.codebook_value(c) for c in codes], np.float32) * np.float32(table[bb])
        np.testing.assert_array_equal(rec, x)


def test_pack_sizes_and_rejections():
    g = load_golden("format_sizes.txt")
    W = tiny_gemv(M=8, K=256)["W"]
    P = oracle.rfp2_pack(W)
    assert P.nbytes == 8 * 256 // g["rfp2_block_weights"] * g["rfp2_block_bytes"]
    assert P.nbytes * 8 / W.size == g["rfp2_bpw"]
    with pytest.raises(ValueError):
        oracle.rfp2_pack(np.zeros((2, 48), np.float32))
    bad = W.copy()
    bad[3, 5] = np.nan
    with pytest.raises(ValueError):
        oracle.rfp2_pack(bad)
    bad[3, 5] = np.inf
    with pytest.raises(ValueError):
        oracle.rfp2_pack(bad)


def test_pack_layout_matches_independent_unpack():
    """Codes read back with an independent unpacker equal per-half code choices."""
    W = decode_gemv(M=4, K=256)["W"]
    P = oracle.rfp2_pack(W)
    codes = unpack_codes(P, 4, 256)
    for m in range(4):
        for h in range(256 // 16):
            b, c = oracle.rfp2_quantize_half(W[m, 16 * h:16 * h + 16])
            np.testing.assert_array_equal(codes[m, 16 * h:16 * h + 16], c)
            assert P[m, h // 2, 8 + h % 2] == b


def test_validate_counts_bad_scale_bytes():
    P = oracle.rfp2_pack(tiny_gemv(M=4, K=64)["W"])
    assert oracle.rfp2_count_bad_scales(P) == 0
    P[1, 0, 9] = 0x7F
    P[2, 1, 8] = 0xFF
    assert oracle.rfp2_count_bad_scales(P) == 2
    with pytest.raises(ValueError):
        oracle.rfp2_decode(P, 4, 64)


# -- activation quantize (Q8_1-style blocks) ----------------------------------

def _independent_quantize(x: np.ndarray):
    x = x.astype(np.float32).reshape(x.shape[0], -1, 32)
    amax = np.abs(x).max(axis=2)
    d = (amax / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (x / d[:, :, None]).astype(np.float32).astype(np.float64)
    q = np.trunc(v + np.copysign(0.5, v))
    q = np.where(d[:, :, None] == 0, 0, np.clip(q, -127, 127))
    return q.reshape(x.shape[0], -1).astype(np.int8), d


def test_quantize_act_hand_cases():
    x = np.zeros((1, 64), np.float32)
    x[0, :4] = [127.0, 2.5, -2.5, -126.5]   # d = 1: halves round away from zero
    x[0, 4] = 0.49999997
    q, d = oracle.quantize_act(x)
    assert d[0, 0] == 1.0 and d[0, 1] == 0.0
    assert list(q[0, :5]) == [127, 3, -3, -127, 0]
    assert np.all(q[0, 32:] == 0)
    # the largest magnitude always maps to +-127
    y = np.random.default_rng(1).normal(0, 3, (3, 96)).astype(np.float32)
    q, d = oracle.quantize_act(y)
    for n in range(3):
        for j in range(3):
            blk = y[n, 32 * j:32 * j + 32]
            i = np.argmax(np.abs(blk))
            assert abs(int(q[n, 32 * j + i])) == 127


def test_quantize_act_matches_independent_numpy():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 1, (4, 1024)), rng.standard_t(3, (2, 1024)) * 1e-3,
                        np.zeros((1, 1024))]).astype(np.float32)
    x[5, 100:140] = 0.0
    q, d = oracle.quantize_act(x)
    qi, di = _independent_quantize(x)
    np.testing.assert_array_equal(d, di)
    np.testing.assert_array_equal(q, qi)


# -- dot products ---------------------------------------------------------------

def test_int_path_matches_brute_force_and_numpy():
    w = tiny_gemv(M=48, K=512, N=3)
    P = oracle.rfp2_pack(w["W"])
    q, d = oracle.quantize_act(w["x"])
    y_int = oracle.rfp2_gemv(P, 48, 512, q, d)
    y_brute = oracle.rfp2_gemv_brute(P, 48, 512, q, d)
    assert np.all(rel_err_rows(y_int, y_brute) <= 1e-12)
    Wd = decode_weights_independent(P, 48, 512)
    a = q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)
    y_np = a @ Wd.T
    assert np.all(rel_err_rows(y_int, y_np) <= 1e-12)


def test_k32_hand_example():
    # one block: codes all 3 (+4) in half 0, all 0 (-4) in half 1
    blk = np.zeros((1, 1, 10), np.uint8)
    blk[0, 0, :4] = 0xFF
    blk[0, 0, 4:8] = 0x00
    blk[0, 0, 8] = 0x38   # 0.5
    blk[0, 0, 9] = 0x40   # (8+0) * 2^(8-11) = 1.0
    q = np.arange(-16, 16, dtype=np.int8).reshape(1, 32)
    d = np.array([[0.25]], np.float32)
    # S0 = 4 * sum(-16..-1) = -544, S1 = -4 * sum(0..15) = -480
    parts = oracle.rfp2_half_partials(blk, 1, 32, q)
    assert list(parts[0, 0]) == [-544, -480]
    y = oracle.rfp2_gemv(blk, 1, 32, q, d)
    assert y[0, 0] == 0.25 * (0.5 * -544 + 1.0 * -480)


def test_half_partials_match_numpy_int_dot():
    w = tiny_gemv(M=16, K=256, N=2)
    P = oracle.rfp2_pack(w["W"])
    q, _ = oracle.quantize_act(w["x"])
    parts = oracle.rfp2_half_partials(P, 16, 256, q)
    levels = np.array([-4, -1, 1, 4], np.int64)[unpack_codes(P, 16, 256)]
    ref = (levels[None, :, :] * q[:, None, :].astype(np.int64)).reshape(2, 16, 16, 16).sum(-1)
    np.testing.assert_array_equal(parts, ref)
    assert np.abs(parts).max() <= 16 * 4 * 127


def test_gemv_row_subset_equals_full():
    w = tiny_gemv(M=32, K=256, N=2)
    P = oracle.rfp2_pack(w["W"])
    q, d = oracle.quantize_act(w["x"])
    full = oracle.rfp2_gemv(P, 32, 256, q, d)
    rows = np.array([31, 0, 7, 7])
    np.testing.assert_array_equal(oracle.rfp2_gemv(P, 32, 256, q, d, rows=rows), full[:, rows])


# -- MoE -------------------------------------------------------------------------

def test_moe_equals_per_expert_gemv():
    E, M, K, T, top_k = 6, 16, 128, 5, 3
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=11)
    P = np.stack([oracle.rfp2_pack(w["W"][e]) for e in range(E)])
    q, d = oracle.quantize_act(w["x"])
    y = oracle.rfp2_moe(P, E, M, K, w["ids"], q, d)
    for t in range(T):
        for j in range(top_k):
            e = w["ids"][t, j]
            ref = oracle.rfp2_gemv(P[e], M, K, q[t:t + 1], d[t:t + 1])
            np.testing.assert_array_equal(y[t, j], ref[0])
    bad = w["ids"].copy()
    bad[2, 1] = E
    with pytest.raises(ValueError):
        oracle.rfp2_moe(P, E, M, K, bad, q, d)
    bad[2, 1] = -1
    with pytest.raises(ValueError):
        oracle.rfp2_moe(P, E, M, K, bad, q, d)


# -- prefill GEMM -------------------------------------------------------------------

def test_gemm_rows_match_numpy_float64():
    import torch
    rng = np.random.default_rng(9)
    M, K, N = 24, 256, 7
    W = rng.normal(0, 0.015, (M, K)).astype(np.float32)
    P = oracle.rfp2_pack(W)
    xf = rng.normal(0, 1, (N, K)).astype(np.float32)
    X = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    Xf = torch.from_numpy(X.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    ref = Xf @ decode_weights_independent(P, M, K).T
    y = oracle.rfp2_gemm(P, M, K, X)
    assert np.all(rel_err_rows(y, ref) <= 1e-12)
    rows = np.array([5, 23])
    np.testing.assert_array_equal(oracle.rfp2_gemm(P, M, K, X, rows=rows), y[:, rows])


def test_synth_bf16_cast_matches_torch():
    import torch
    from synth import float32_to_bf16_bits
    x = np.random.default_rng(3).normal(0, 1, 4096).astype(np.float32) * 20
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(float32_to_bf16_bits(x), ref)


# -- importance-weighted scale search ("05 Completed experiment") ----------------

def _ue4m3_values():
    return [oracle.ue4m3(b) for b in range(0x7F)]


def test_weighted_pack_equals_plain_pack_for_flat_blocks():
    """With importance 1 and every |x| of a block equal, each term's weight
    importance * sqrt(sigma^2 + x^2) is one constant per block, so the
    weighted search has the plain search's minimiser."""
    rng = np.random.default_rng(11)
    M, K = 6, 256
    mags = np.repeat(rng.uniform(1e-3, 0.3, (M, K // 32)), 32, axis=1)
    W = (mags * rng.choice([-1.0, 1.0], (M, K))).astype(np.float32)
    P = oracle.rfp2_pack_weighted(W, np.ones(K, np.float32))
    np.testing.assert_array_equal(P, oracle.rfp2_pack(W))


def test_weighted_pack_is_invariant_to_power_of_two_importance_scaling():
    from synth import imatrix_importance
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((5, 512)) * 0.02).astype(np.float32)
    imp = imatrix_importance(512)
    P = oracle.rfp2_pack_weighted(W, imp)
    for k in (-20, -3, 5):
        np.testing.assert_array_equal(oracle.rfp2_pack_weighted(W, np.ldexp(imp, k)), P)


def test_weighted_pack_one_hot_importance_makes_that_weight_exact():
    """All importance on one weight of each half: the objective is zero exactly
    at the bytes whose level grid holds that weight, so the smallest such byte
    wins."""
    scales = _ue4m3_values()
    rng = np.random.default_rng(13)
    K = 64
    W = (rng.standard_normal((1, K)) * 0.05).astype(np.float32)
    imp = np.zeros(K, np.float32)
    targets = {}
    for h in range(K // 16):
        i0 = 16 * h + int(rng.integers(16))
        b0 = int(rng.integers(8, 0x7F))
        W[0, i0] = np.float32(rng.choice([-4.0, -1.0, 1.0, 4.0]) * scales[b0])
        imp[i0] = 1.0
        x = float(W[0, i0])
        zero = [b for b in range(0x7F) if scales[b] > 0 and
                (abs(x) == scales[b] or abs(x) == 4 * scales[b])]
        targets[h] = min(zero)
    P = oracle.rfp2_pack_weighted(W, imp)
    for h, b in targets.items():
        assert P[0, h // 2, 8 + h % 2] == b


def test_weighted_pack_zero_importance_picks_the_first_byte():
    W = (np.random.default_rng(14).standard_normal((2, 64)) * 0.1).astype(np.float32)
    P = oracle.rfp2_pack_weighted(W, np.zeros(64, np.float32))
    assert np.all(P[..., 8:] == 0)


def test_weighted_pack_never_loses_on_its_own_objective():
    """Per half, the weighted search's choice has a weighted error no larger
    than the plain search's choice (and the plain choice is likewise never
    worse on the plain error)."""
    from synth import imatrix_importance
    rng = np.random.default_rng(15)
    M, K = 4, 256
    W = (rng.standard_t(5, (M, K)) * 0.02).astype(np.float32)
    imp = imatrix_importance(K)
    Pw, Pp = oracle.rfp2_pack_weighted(W, imp), oracle.rfp2_pack(W)
    better = 0
    for m in range(M):
        for j in range(K // 32):
            x32 = W[m, 32 * j:32 * j + 32]
            s2 = oracle.rfp2_block_sigma2(x32)
            acc = 0.0
            for v in x32.astype(np.float64):
                acc += v * v
            assert s2 == 2.0 * acc / 32.0
            for h in range(2):
                x, w = x32[16 * h:16 * h + 16], imp[32 * j + 16 * h:32 * j + 16 * h + 16]
                ew = oracle.rfp2_half_wsse(x, w, s2, int(Pw[m, j, 8 + h]))
                ep = oracle.rfp2_half_wsse(x, w, s2, int(Pp[m, j, 8 + h]))
                assert ew <= ep
                better += ew < ep
    assert better > 0


def _weighted_golden_block():
    g = load_golden("rfp2_weighted_objective.txt")
    x = np.zeros(32, np.float32)
    imp = np.zeros(32, np.float32)
    cols = [int(c) for c in g["nonzero_columns"]]
    x[cols] = g["nonzero_values"]
    imp[cols] = g["importance"]
    return g, x, imp


def test_weighted_objective_golden_block():
    """The hand-derived block of the golden fixture: sigma^2, the objective's
    closed-form values at the two contending bytes of each half, and the
    packed block (0x3F for half 0, 0x40 for half 1) all follow the page's
    weight importance * sqrt(sigma^2 + x^2); dropping the square root,
    squaring the importance or dropping sigma^2 would pick other bytes."""
    g, x, imp = _weighted_golden_block()
    s2 = oracle.rfp2_block_sigma2(x)
    assert s2 == g["sigma2"]
    ra, rb = math.sqrt(s2 + 1.0), math.sqrt(s2 + 14.0625)
    for h, ia in ((0, 16.0), (1, 48.0)):
        xs, ws = x[16 * h:16 * h + 16], imp[16 * h:16 * h + 16]
        assert math.isclose(oracle.rfp2_half_wsse(xs, ws, s2, 0x3F), ia * ra / 256, rel_tol=1e-14)
        assert math.isclose(oracle.rfp2_half_wsse(xs, ws, s2, 0x40), rb / 16, rel_tol=1e-14)
    P = oracle.rfp2_pack_weighted(x.reshape(1, 32), imp)
    assert [int(v) for v in P.ravel()] == [int(v) for v in g["block"]]
    assert [int(v) for v in P.ravel()[8:]] == [int(v) for v in g["bytes_page_formula"]]


def test_weighted_objective_golden_block_separates_mistaken_weights():
    """The fixture discriminates: an independent brute force over the 127
    scale bytes (UE4M3 from torch's E4M3FN decoder, halved) reproduces the
    fixture's bytes for the page's weight and for each mistaken form, and
    every mistaken form's bytes differ from the page formula's."""
    g, x, imp = _weighted_golden_block()
    table = e4m3fn_half_table()
    s2 = float(g["sigma2"])
    forms = {
        "bytes_page_formula": lambda i, v: i * math.sqrt(s2 + v * v),
        "bytes_without_sqrt": lambda i, v: i * (s2 + v * v),
        "bytes_importance_squared": lambda i, v: i * i * math.sqrt(s2 + v * v),
        "bytes_without_sigma2": lambda i, v: i * abs(v),
    }
    for key, wfun in forms.items():
        got = []
        for h in range(2):
            xs, ws = x[16 * h:16 * h + 16].astype(np.float64), imp[16 * h:16 * h + 16]
            best = None
            for b in range(0x7F):
                s = float(table[b])
                err = 0.0
                for v, i in zip(xs, ws):
                    inner = s == 0.0 or abs(np.float32(v) / np.float32(s)) <= 2.5
                    r = 0.0 if s == 0.0 else (1.0 if inner else 4.0) * s * (-1.0 if v < 0 else 1.0)
                    err += wfun(float(i), float(v)) * (v - r) ** 2
                if best is None or err < best[0]:
                    best = (err, b)
            got.append(best[1])
        assert got == [int(v) for v in g[key]], key
        if key != "bytes_page_formula":
            assert got != [int(v) for v in g["bytes_page_formula"]], key
