"""GPU parity of the activation quantizer, the packers, the int32 half sums and
the dense ROCmFP2 GEMV against the CPU oracle, through the C ABI.

Bar (statement of the problem): packed bytes, int8 activations, their scales
and every int32 half sum bit-exact; fp32 outputs within 1e-5 relative,
normwise per output row (one token's [M] vector), of the fp64 oracle.
"""
import numpy as np
import pytest

import oracle
from synth import child_rngs, decode_gemv, hfp4_gemv, normal_weights, tiny_gemv
from _helpers import rel_err_rows, rows_parallel

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def g():
    import gemm_rocmfp2_mul_gb300 as g
    g.build()
    g.lib()
    return g


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.cpu().numpy()


def status_tensor():
    import torch
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _inputs(kind, N, K, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        x = rng.normal(0, 1, (N, K))
    elif kind == "student_t":
        x = rng.standard_t(3, (N, K)) * 1e-3
    elif kind == "wide":
        x = rng.normal(0, 1, (N, K)) * 10.0 ** rng.integers(-6, 6, (N, K // 32, 1)).repeat(32, 2).reshape(N, K)
    elif kind == "ties":
        # a / d within a few ulps of a half-integer, for scales d that are
        # not powers of two: the rounding decision sits at its boundary
        d = (rng.random((N, K // 32, 1)) + 0.5).astype(np.float32)
        k = rng.integers(-127, 127, (N, K // 32, 32)).astype(np.float32) + 0.5
        x = (k * d).astype(np.float32)
        ulps = rng.integers(-3, 4, x.shape)
        x = np.nextafter(x, np.where(ulps > 0, np.inf, -np.inf).astype(np.float32)) * (ulps != 0) + x * (ulps == 0)
        x[:, :, 0] = 127.0 * d[:, :, 0]
        x = x.reshape(N, K)
    elif kind == "near_half":
        # a within 16 float steps of (k + 1/2) * d0 for scales over 120
        # binades, block max 127 * d0: exercises the kernel's exact
        # near-half rounding on both sides of every boundary
        d0 = (rng.uniform(1, 2, (N, K // 32, 1)) * np.exp2(rng.integers(-60, 60, (N, K // 32, 1))))
        d0 = d0.astype(np.float32)
        k = rng.integers(-127, 127, (N, K // 32, 32)).astype(np.float32) + np.float32(0.5)
        x = (k * d0).astype(np.float32)
        step = rng.integers(-16, 17, x.shape).astype(np.int32)
        x = (x.view(np.int32) + step).view(np.float32)
        x[:, :, 0] = np.float32(127) * d0[:, :, 0]
        x = x.reshape(N, K)
    elif kind == "subnormal":
        # block maxima near and below the smallest normal: d is subnormal
        x = rng.normal(0, 1, (N, K)) * 10.0 ** rng.integers(-44, -36, (N, K // 32, 1)).repeat(32, 2).reshape(N, K)
    else:
        x = rng.normal(0, 1, (N, K))
        x[:, :64] = 0.0
        x[:, 64:96] = -0.0
        # exact halves: block max 127 -> d = 1, values k + 0.5 tie away from zero
        x[:, 96:128] = np.arange(-16, 16) + 0.5
        x[:, 127] = 127.0
    return x.astype(np.float32)


# -- activation quantization ------------------------------------------------------

KINDS = ["normal", "student_t", "wide", "edge", "ties", "near_half", "subnormal"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("N,K", [(1, 4096), (4, 2048), (8, 256), (3, 8192)])
def test_quantize_bit_exact(g, kind, N, K):
    x = _inputs(kind, N, K, seed=N * K)
    q, d = g.rfp2_quantize_act(dev(x))
    qo, do = oracle.quantize_act(x)
    np.testing.assert_array_equal(host(d), do)
    np.testing.assert_array_equal(host(q), qo)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("N,K", [(1, 4096), (2, 2048), (1, 256), (2, 16384), (3, 4096), (4, 1024),
                                 (8, 512)])
def test_gemv_quantize_bit_exact(g, kind, N, K):
    """rfp2_gemv quantizes inside the GEMV kernel at batch <= 8; the q and d it
    leaves in the workspace are the oracle's, bit for bit (the "ties" kind puts
    a/d within a few ulps of half-integers, where the kernel decides the
    rounding by an exact comparison instead of the division)."""
    import torch
    x = _inputs(kind, N, K, seed=7 * N + K)
    W = normal_weights(np.random.default_rng(K), 160, K, 0.02)
    P = oracle.rfp2_pack(W)
    ws = torch.zeros(g.rfp2_gemv_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    y = host(g.rfp2_gemv(dev(P), 160, K, dev(x), workspace=ws, dev_status=st))
    assert host(st)[0] == 0
    qo, do = oracle.quantize_act(x)
    wsh = host(ws)
    np.testing.assert_array_equal(wsh[:N * K].view(np.int8).reshape(N, K), qo)
    off = (N * K + 255) // 256 * 256
    np.testing.assert_array_equal(wsh[off:off + N * K // 32 * 4].view(np.float32).reshape(N, -1), do)
    ref = oracle.rfp2_gemv(P, 160, K, qo, do)
    if np.all(np.abs(ref).max(axis=1) > 0):
        assert np.all(rel_err_rows(y, ref) <= TOL)


# -- packers ------------------------------------------------------------------------

def _weights(kind, M, K, seed=0):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        W = rng.normal(0, 0.02, (M, K))
    elif kind == "student_t":
        W = rng.standard_t(5, (M, K)) * 0.02
        W[:, rng.choice(K, max(1, K // 100), replace=False)] *= 8
    elif kind == "tiny":
        W = rng.normal(0, 1e-5, (M, K))
    elif kind == "huge":
        W = rng.normal(0, 100.0, (M, K))
    else:
        W = rng.normal(0, 0.5, (M, K)) * (rng.random((M, K)) < 0.3)
        W[0, :32] = 0.0
        W[1, :32] = -0.0
    return W.astype(np.float32)


@pytest.mark.parametrize("kind", ["normal", "student_t", "tiny", "huge", "sparse"])
def test_rfp2_pack_bit_exact(g, kind):
    W = _weights(kind, 64, 512, seed=3)
    P = host(g.rfp2_pack_weights(dev(W)))
    np.testing.assert_array_equal(P, oracle.rfp2_pack(W))


def test_rfp2_pack_tiny_config_bit_exact(g):
    W = tiny_gemv()["W"]   # 256 x 1024, seed 0
    np.testing.assert_array_equal(host(g.rfp2_pack_weights(dev(W))), oracle.rfp2_pack(W))


@pytest.mark.parametrize("kind", ["normal", "student_t", "tiny", "huge", "sparse"])
def test_rfp2_pack_weighted_bit_exact(g, kind):
    """Importance-weighted scale search ("05 Completed experiment"): packed
    bytes equal the oracle's, with synthetic importance, one-hot importance
    and all-zero importance."""
    from synth import imatrix_importance
    W = _weights(kind, 48, 512, seed=21)
    imp = imatrix_importance(512)
    for importance in (imp, np.eye(1, 512, 37, dtype=np.float32).ravel() * 3.0,
                       np.zeros(512, np.float32)):
        Pg = g.rfp2_pack_weights_weighted(dev(W), dev(importance.astype(np.float32)))
        np.testing.assert_array_equal(host(Pg), oracle.rfp2_pack_weighted(W, importance))


@pytest.mark.parametrize("kind", ["normal", "student_t", "tiny", "huge", "sparse"])
def test_hfp4_pack_bit_exact(g, kind):
    W = _weights(kind, 48, 1024, seed=5)
    st = status_tensor()
    P = host(g.hfp4_pack_weights(dev(W), dev_status=st))
    assert host(st)[0] == 0
    np.testing.assert_array_equal(P, oracle.hfp4_pack(W))


# -- int32 half sums ------------------------------------------------------------------

def test_half_partials_bit_exact(g):
    w = tiny_gemv(M=96, K=512, N=5, seed=7)
    P = oracle.rfp2_pack(w["W"])
    q, _ = oracle.quantize_act(w["x"])
    got = host(g.rfp2_debug_half_partials(dev(P), 96, 512, dev(q)))
    np.testing.assert_array_equal(got, oracle.rfp2_half_partials(P, 96, 512, q))


def test_half_partials_extremes_bit_exact(g):
    # +-127 activations against all-outer levels reach |S| = 16*4*127
    rng = np.random.default_rng(1)
    P = rng.integers(0, 256, (8, 4, 10)).astype(np.uint8)
    P[:, :, 8:] = rng.integers(0, 0x7F, (8, 4, 2))
    P[0, :, :8] = 0xFF
    P[1, :, :8] = 0x00
    q = rng.integers(-127, 128, (3, 128)).astype(np.int8)
    q[0] = 127
    q[1] = -127
    got = host(g.rfp2_debug_half_partials(dev(P), 8, 128, dev(q)))
    ref = oracle.rfp2_half_partials(P, 8, 128, q)
    np.testing.assert_array_equal(got, ref)
    assert np.abs(ref).max() == 16 * 4 * 127


# -- dense GEMV ------------------------------------------------------------------------

def _gemv_case(g, M, K, N, seed, fused=True):
    rng = child_rngs(seed, 2)
    W = normal_weights(rng[0], M, K, 0.02)
    x = rng[1].standard_normal((N, K)).astype(np.float32)
    P = oracle.rfp2_pack(W)
    q, d = oracle.quantize_act(x)
    ref = oracle.rfp2_gemv(P, M, K, q, d)
    st = status_tensor()
    if fused:
        import torch
        ws = torch.empty(g.rfp2_gemv_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
        y = host(g.rfp2_gemv(dev(P), M, K, dev(x), workspace=ws, dev_status=st))
        wsh = host(ws)
        np.testing.assert_array_equal(wsh[:N * K].view(np.int8).reshape(N, K), q)
        off = (N * K + 255) // 256 * 256
        np.testing.assert_array_equal(wsh[off:off + N * K // 32 * 4].view(np.float32).reshape(N, -1), d)
    else:
        y = host(g.rfp2_gemv_q8(dev(P), M, K, dev(q), dev(d), dev_status=st))
    assert host(st)[0] == 0
    return y, ref


@pytest.mark.parametrize("M,K,N", [
    (256, 1024, 1), (1000, 4096, 1), (1000, 4096, 4), (777, 2048, 3), (64, 256, 8),
    (333, 8192, 2), (50, 5120, 4), (130, 768, 5), (300, 1536, 6), (129, 2048, 7),
    (1, 4096, 8), (5, 256, 1), (2048, 4096, 2), (64, 16384, 1), (40, 32768, 2),
])
def test_gemv_parity(g, M, K, N):
    y, ref = _gemv_case(g, M, K, N, seed=M + K + N)
    err = rel_err_rows(y, ref)
    assert np.all(err <= TOL), err.max()


@pytest.mark.parametrize("M,K,N", [(640, 4096, 1), (640, 4096, 4), (100, 2048, 8)])
def test_gemv_q8_parity(g, M, K, N):
    y, ref = _gemv_case(g, M, K, N, seed=11, fused=False)
    assert np.all(rel_err_rows(y, ref) <= TOL)


def test_gemv_max_k(g):
    # K = 65536 at batch 1: every row is split over all sixteen consumer warps
    y, ref = _gemv_case(g, 24, 65536, 1, seed=2)
    assert np.all(rel_err_rows(y, ref) <= TOL)


@pytest.mark.parametrize("M,K,N,fused", [(24, 65536, 8, True), (70, 32768, 7, True),
                                         (33, 65536, 3, False)])
def test_gemv_column_groups(g, M, K, N, fused):
    """Long rows at several columns: the quantized activations of all columns
    do not fit in shared memory, so the columns run in groups (one launch
    each); q/d in the workspace and every output row still match."""
    y, ref = _gemv_case(g, M, K, N, seed=M + N, fused=fused)
    assert np.all(rel_err_rows(y, ref) <= TOL)


def test_gemv_tiny_config(g):
    """256 x 1024 N(0, 0.02^2) weights, one N(0,1) vector, seed 0."""
    w = tiny_gemv()
    P = oracle.rfp2_pack(w["W"])
    q, d = oracle.quantize_act(w["x"])
    ref = oracle.rfp2_gemv(P, 256, 1024, q, d)
    Pg = g.rfp2_pack_weights(dev(w["W"]))
    np.testing.assert_array_equal(host(Pg), P)
    y = host(g.rfp2_gemv(Pg, 256, 1024, dev(w["x"])))
    assert np.all(rel_err_rows(y, ref) <= TOL)
    # the brute-force fp64 formulation agrees too
    assert np.all(rel_err_rows(y, oracle.rfp2_gemv_brute(P, 256, 1024, q, d)) <= TOL)


@pytest.fixture(scope="module")
def decode_full(g):
    w = decode_gemv(N=8)   # 14336 x 4096, Student-t(5)*0.02, 41 outlier columns x8, seed 1
    Pg = g.rfp2_pack_weights(dev(w["W"]))
    Po = rows_parallel(oracle.rfp2_pack, w["W"])   # every row, on all host cores
    return w, Pg, Po


def test_decode_full_size_packing_bit_exact(g, decode_full):
    """The GPU packer reproduces every one of the 18,350,080 bytes of the
    oracle's packing of the 14336 x 4096 decode weights."""
    w, Pg, Po = decode_full
    np.testing.assert_array_equal(host(Pg), Po)


@pytest.mark.parametrize("N", [1, 3, 4, 8])
def test_decode_full_size(g, decode_full, N):
    """Full 14336 x 4096 decode GEMV in the benchmark's launch configuration,
    every output row checked against the oracle (normwise per token over all
    14336 rows, and elementwise against the sum of absolute terms)."""
    import torch
    w, Pg, Po = decode_full
    M, K = w["W"].shape
    x = w["x"][:N]
    ws = torch.empty(g.rfp2_gemv_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    st = status_tensor()
    y = host(g.rfp2_gemv(Pg, M, K, dev(x), workspace=ws, dev_status=st))
    assert host(st)[0] == 0
    q, d = oracle.quantize_act(x)
    ref = rows_parallel(lambda P, q, d: oracle.rfp2_gemv(P, P.shape[0], K, q, d).T, Po, q, d).T
    assert np.all(rel_err_rows(y, ref) <= TOL)
    Wd = oracle.rfp2_decode(Po, M, K).astype(np.float64)
    a = q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)
    bound = np.abs(a) @ np.abs(Wd).T
    assert np.all(np.abs(y - ref) <= TOL * bound)


def test_zero_inputs_give_exact_zero(g):
    W = normal_weights(np.random.default_rng(0), 64, 512, 0.02)
    P = oracle.rfp2_pack(W)
    y = host(g.rfp2_gemv(dev(P), 64, 512, dev(np.zeros((2, 512), np.float32))))
    assert np.all(y == 0.0)
    Pz = oracle.rfp2_pack(np.zeros((16, 512), np.float32))
    y = host(g.rfp2_gemv(dev(Pz), 16, 512, dev(np.ones((3, 512), np.float32))))
    assert np.all(y == 0.0)


def test_deterministic(g):
    w = tiny_gemv(M=512, K=2048, N=4, seed=9)
    P = dev(oracle.rfp2_pack(w["W"]))
    y1 = host(g.rfp2_gemv(P, 512, 2048, dev(w["x"])))
    y2 = host(g.rfp2_gemv(P, 512, 2048, dev(w["x"])))
    np.testing.assert_array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_error_codes(g):
    import torch
    P = dev(np.zeros((8, 512 // 32, 10), np.uint8))
    x = dev(np.zeros((1, 512), np.float32))
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv(dev(np.zeros((8, 3, 10), np.uint8)), 8, 96, dev(np.zeros((1, 96), np.float32)))
    assert e.value.status == 4   # K % 256 -> unsupported on the GPU
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv(P, 8, 512, dev(np.zeros((9, 512), np.float32)))
    assert e.value.status == 2   # N > 8
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv(P, 8, 512, x, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 9   # workspace too small
    raw = torch.zeros(8 * 160 + 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv(raw[1:1 + 8 * 160], 8, 512, x)
    assert e.value.status == 3   # weights not 16-byte aligned


def test_validate_weights(g):
    P = oracle.rfp2_pack(tiny_gemv(M=32, K=256)["W"])
    st = status_tensor()
    assert int(host(g.rfp2_validate_weights(dev(P), dev_status=st))[0]) == 0
    assert host(st)[0] == 0
    P[3, 2, 8] = 0x7F
    P[7, 0, 9] = 0xC0
    P[31, 7, 9] = 0xFF
    bad = host(g.rfp2_validate_weights(dev(P), dev_status=st))
    assert int(bad[0]) == 3 == oracle.rfp2_count_bad_scales(P)
    assert host(st)[0] == 6   # RFP2_EBADSCALE


def test_gemv_right_after_packing_on_the_same_stream(g):
    """Weight prefetch is off by default: rfp2_gemv enqueued right after
    rfp2_pack_weights on the same stream, with no synchronization between
    them, reads the freshly packed weights (the destination starts as 0xFF
    bytes, whose scale bytes are illegal, so stale bytes would show)."""
    import torch
    assert not g.rfp2_weight_prefetch()
    M, K, N = 2048, 4096, 1
    r_w, r_x = child_rngs(321, 2)
    W = normal_weights(r_w, M, K, 0.02)
    x = r_x.standard_normal((N, K)).astype(np.float32)
    Wd, xd = dev(W), dev(x)
    torch.cuda.synchronize()
    P = torch.full((M, K // 32, 10), 0xFF, dtype=torch.uint8, device="cuda")
    g.rfp2_pack_weights(Wd, out=P)
    y = host(g.rfp2_gemv(P, M, K, xd))
    Po = oracle.rfp2_pack(W)
    q, d = oracle.quantize_act(x)
    assert np.all(rel_err_rows(y, oracle.rfp2_gemv(Po, M, K, q, d)) <= TOL)


@pytest.mark.parametrize("N", [1, 2, 4])
def test_gemv_with_weight_prefetch(g, N):
    """With rfp2_set_weight_prefetch(1) the GEMV streams W before the
    previous kernel on the stream has completed (the weights here were
    written and synchronized before); back-to-back calls on two weight
    matrices still match the oracle."""
    import torch
    M, K = 1500, 4096
    rng = child_rngs(400 + N, 4)
    Ws = [normal_weights(rng[i], M, K, 0.02) for i in range(2)]
    xs = [rng[2 + i].standard_normal((N, K)).astype(np.float32) for i in range(2)]
    Ps = [oracle.rfp2_pack(W) for W in Ws]
    Pd = [dev(P) for P in Ps]
    xd = [dev(x) for x in xs]
    torch.cuda.synchronize()
    g.rfp2_set_weight_prefetch(True)
    try:
        ys = [g.rfp2_gemv(Pd[i % 2], M, K, xd[(i // 2) % 2]) for i in range(4)]
        torch.cuda.synchronize()
    finally:
        g.rfp2_set_weight_prefetch(False)
    for i, y in enumerate(ys):
        q, d = oracle.quantize_act(xs[(i // 2) % 2])
        ref = oracle.rfp2_gemv(Ps[i % 2], M, K, q, d)
        assert np.all(rel_err_rows(host(y), ref) <= TOL)
