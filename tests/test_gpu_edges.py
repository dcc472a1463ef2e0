"""Edge cases of every entry point, through the C ABI on the GPU: empty and
out-of-range sizes (the documented status, no launch), ragged shapes that
leave partial tiles, the largest supported batch, and the degenerate inputs
the method has (all-zero weights or activations give exact zeros; one-token,
one-expert routing)."""
import ctypes as C

import numpy as np
import pytest

import oracle
from synth import child_rngs, float32_to_bf16_bits, normal_weights
from _helpers import rel_err_rows

pytestmark = pytest.mark.gpu
OK, EINVAL, ESHAPE, EUNSUPPORTED = 0, 1, 2, 4


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


@pytest.fixture(scope="module")
def buf():
    import torch
    return torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")


def test_empty_and_out_of_range_sizes(g, buf):
    L = g.lib()
    p = C.c_void_p(buf.data_ptr())
    n = len(buf)
    # quantize and packers: zero rows or columns are a no-op
    assert L.rfp2_quantize_act(p, 0, 256, p, p, None) == OK
    assert L.rfp2_quantize_act(p, 3, 0, p, p, None) == OK
    assert L.rfp2_quantize_act(p, 1, 100, p, p, None) == ESHAPE
    assert L.rfp2_quantize_act(p, -1, 256, p, p, None) == EINVAL
    assert L.rfp2_pack_weights(p, 0, 256, p, None) == OK
    assert L.rfp2_pack_weights(p, 4, 100, p, None) == ESHAPE
    assert L.rfp2_pack_weights_weighted(p, 0, 256, p, p, None) == OK
    assert L.hfp4_pack_weights(p, 0, 256, p, None, None) == OK
    # products: a zero-sized operand or a batch outside [1, 8] is a shape error
    for M, K, N in ((0, 256, 1), (16, 0, 1), (16, 256, 0), (16, 256, 9)):
        assert L.rfp2_gemv_q8(p, M, K, p, p, N, p, None, None) == ESHAPE
        assert L.rfp2_gemv(p, M, K, p, N, p, p, n, None, None) == ESHAPE
        assert L.hfp4_gemv(p, M, K, p, N, p, p, n, None, None) == ESHAPE
    assert L.rfp2_gemv(p, 16, 128, p, 1, p, p, n, None, None) == EUNSUPPORTED
    for M, K, N in ((0, 256, 4), (16, 0, 4), (16, 256, 0)):
        assert L.rfp2_gemm(p, M, K, p, N, p, p, n, None, None) == ESHAPE
        assert L.hfp4_gemm(p, M, K, p, N, p, p, n, None, None) == ESHAPE
        assert L.rfp2_gemv_batched(p, M, K, p, N, p, p, n, None, None) == ESHAPE
    for E, M, K, T, top_k in ((0, 16, 256, 1, 1), (4, 0, 256, 1, 1), (4, 16, 256, 0, 1),
                              (4, 16, 256, 1, 0)):
        assert L.rfp2_moe_gemv(p, E, M, K, p, T, top_k, p, p, p, n, None, None) == ESHAPE


def _gemv_case(g, M, K, N, seed):
    rw, rx = child_rngs(seed, 2)
    W = normal_weights(rw, M, K, 0.02)
    x = rx.standard_normal((N, K)).astype(np.float32)
    P = oracle.rfp2_pack(W)
    q, d = oracle.quantize_act(x)
    return P, x, oracle.rfp2_gemv(P, M, K, q, d)


@pytest.mark.parametrize("M", [1, 3, 17, 95, 153, 305])
@pytest.mark.parametrize("N", [1, 3, 8])
def test_gemv_ragged_rows_and_largest_batch(g, M, N):
    P, x, ref = _gemv_case(g, M, 512, N, seed=M * 10 + N)
    y = host(g.rfp2_gemv(dev(P), M, 512, dev(x)))
    assert np.all(rel_err_rows(y, ref) <= 1e-5)


@pytest.mark.parametrize("M,N", [(16, 1), (144, 33), (16, 200)])
def test_verify_batch_ragged(g, M, N):
    P, x, ref = _gemv_case(g, M, 256, N, seed=M + N)
    y = host(g.rfp2_gemv_batched(dev(P), M, 256, dev(x)))
    assert np.all(rel_err_rows(y, ref) <= 1e-5)


@pytest.mark.parametrize("M", [1, 17, 100])
def test_hfp4_gemv_ragged_rows(g, M):
    rw, rx = child_rngs(M, 2)
    P = oracle.hfp4_pack(normal_weights(rw, M, 512, 0.02))
    x = rx.standard_normal((2, 512)).astype(np.float32)
    y = host(g.hfp4_gemv(dev(P), M, 512, dev(x)))
    assert np.all(rel_err_rows(y, oracle.hfp4_gemv(P, M, 512, x)) <= 1e-5)


@pytest.mark.parametrize("hfp4", [False, True])
@pytest.mark.parametrize("M,N", [(16, 1), (272, 129)])
def test_prefill_ragged_tiles(g, hfp4, M, N):
    rw, rx = child_rngs(M + N, 2)
    W = normal_weights(rw, M, 256, 0.02)
    X = float32_to_bf16_bits(rx.standard_normal((N, 256)).astype(np.float32))
    if hfp4:
        P = oracle.hfp4_pack(W)
        Y, ref = host(g.hfp4_gemm(dev(P), M, 256, dev(X.view(np.int16)))), oracle.hfp4_gemm(P, M, 256, X)
    else:
        P = oracle.rfp2_pack(W)
        Y, ref = host(g.rfp2_gemm(dev(P), M, 256, dev(X.view(np.int16)))), oracle.rfp2_gemm(P, M, 256, X)
    assert np.all(rel_err_rows(Y, ref) <= 2e-3)


def test_zero_operands_give_exact_zeros(g):
    M, K, N = 32, 512, 4
    Pz = oracle.rfp2_pack(np.zeros((M, K), np.float32))
    Hz = oracle.hfp4_pack(np.zeros((M, K), np.float32))
    W = normal_weights(np.random.default_rng(1), M, K, 0.02)
    P, H = oracle.rfp2_pack(W), oracle.hfp4_pack(W)
    x = np.random.default_rng(2).standard_normal((N, K)).astype(np.float32)
    zx = np.zeros((N, K), np.float32)
    Xb, Zb = float32_to_bf16_bits(x).view(np.int16), np.zeros((N, K), np.int16)
    outs = [
        g.rfp2_gemv(dev(Pz), M, K, dev(x)), g.rfp2_gemv(dev(P), M, K, dev(zx)),
        g.rfp2_gemv_batched(dev(Pz), M, K, dev(x)), g.rfp2_gemv_batched(dev(P), M, K, dev(zx)),
        g.hfp4_gemv(dev(Hz), M, K, dev(x)), g.hfp4_gemv(dev(H), M, K, dev(zx)),
        g.rfp2_gemm(dev(Pz), M, K, dev(Xb)), g.rfp2_gemm(dev(P), M, K, dev(Zb)),
        g.hfp4_gemm(dev(Hz), M, K, dev(Xb)), g.hfp4_gemm(dev(H), M, K, dev(Zb)),
    ]
    for o in outs:
        assert np.all(host(o) == 0.0)


@pytest.mark.parametrize("E,T,top_k", [(1, 1, 1), (3, 5, 2), (2, 7, 2)])
def test_moe_degenerate_routing(g, E, T, top_k):
    """One expert and one token; every token on the same pair of experts."""
    import torch
    M, K = 96, 256
    rng = np.random.default_rng(E * 10 + T)
    W = np.stack([normal_weights(rng, M, K, 0.02) for _ in range(E)])
    P = np.stack([oracle.rfp2_pack(W[e]) for e in range(E)])
    x = rng.standard_normal((T, K)).astype(np.float32)
    ids = np.tile(np.arange(top_k, dtype=np.int32) % E, (T, 1))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.rfp2_moe_gemv(dev(P), E, M, K, dev(ids), dev(x), dev_status=st))
    assert int(host(st)[0]) == 0
    q, d = oracle.quantize_act(x)
    ref = oracle.rfp2_moe(P, E, M, K, ids, q, d)
    assert np.all(rel_err_rows(y.reshape(T * top_k, M), ref.reshape(T * top_k, M)) <= 1e-5)


def test_bounded_wait_reports_timeout_and_context_survives(g):
    """A wait on an mbarrier that nothing arrives on gives up after the
    library's limit and reports RFP2_ETIMEOUT; the next call runs normally."""
    import time
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    g.rfp2_debug_wait_timeout(st)
    assert int(host(st)[0]) == 8  # RFP2_ETIMEOUT
    assert 1.0 < time.time() - t0 < 30.0
    P, x, ref = _gemv_case(g, 96, 512, 1, seed=5)
    y = host(g.rfp2_gemv(dev(P), 96, 512, dev(x)))
    assert np.all(rel_err_rows(y, ref) <= 1e-5)
