"""GPU parity of the prefill GEMM (rfp2_gemm, tcgen05 tensor cores) against
the CPU oracle, through the C ABI: Y = X W^T with the ROCmFP2 weights decoded
exactly to bf16 inside the kernel; outputs within 2e-3 relative, normwise per
output row (one token's [M] vector), of the fp64 oracle; the decoded weights
bit-exact (one-hot tokens read them back)."""
import numpy as np
import pytest

import oracle
from synth import child_rngs, float32_to_bf16_bits, normal_weights, prefill_gemm
from _helpers import decode_weights_independent, rel_err_rows, rows_parallel

pytestmark = pytest.mark.gpu
TOL = 2e-3


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


def _case(g, M, K, N, seed):
    import torch
    r_w, r_x = child_rngs(seed, 2)
    W = normal_weights(r_w, M, K, 0.015)
    X = float32_to_bf16_bits(r_x.standard_normal((N, K)).astype(np.float32))
    P = oracle.rfp2_pack(W)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = host(g.rfp2_gemm(dev(P), M, K, dev(X.view(np.int16)), dev_status=st))
    assert int(host(st)[0]) == 0
    return Y, P, X


def test_gemm_single_tile(g):
    M, K, N = 256, 256, 128
    Y, P, X = _case(g, M, K, N, seed=1)
    ref = oracle.rfp2_gemm(P, M, K, X)
    assert np.all(rel_err_rows(Y, ref) <= TOL)


@pytest.mark.parametrize("M,K", [(512, 512), (2560, 1024)])
def test_gemm_decoded_weights_exact(g, M, K):
    """Tokens e_k (one-hot bf16 rows) read the in-kernel decode back: Y[k, m]
    = w[m, k] with a single exact product per output, so Y equals the
    oracle's decoded weights bit for bit (both CTAs of a pair, every 16-byte
    chunk of the 128-byte swizzle rows, all four K slices of a packed box;
    512 x 512 runs as quarter tiles only, 2560 x 1024 as 40 whole tiles)."""
    W = normal_weights(child_rngs(11, 1)[0], M, K, 0.015)
    P = oracle.rfp2_pack(W)
    X = np.zeros((K, K), np.uint16)
    X[np.arange(K), np.arange(K)] = 0x3F80  # bf16 1.0
    Y = host(g.rfp2_gemm(dev(P), M, K, dev(X.view(np.int16))))
    np.testing.assert_array_equal(Y, oracle.rfp2_decode(P, M, K).T.astype(np.float32))


@pytest.mark.parametrize("M,K,N", [
    (512, 1024, 256), (272, 768, 200), (1024, 2048, 130), (256, 5120, 7), (4096, 512, 1000),
    # 90 tiles of 256 tokens x 256 weight rows: the 14 past the first wave of
    # 76 CTA pairs run as quarter tiles (N = 64), the last weight tile (16 valid
    # rows) among them; 30 tiles: all as half tiles (N = 128)
    (4368, 256, 1100), (2560, 256, 768),
])
def test_gemm_parity(g, M, K, N):
    Y, P, X = _case(g, M, K, N, seed=M + N + K)
    ref = oracle.rfp2_gemm(P, M, K, X)
    err = rel_err_rows(Y, ref)
    assert np.all(err <= TOL), err.max()
    # the products are exact and the sums fp32: far inside the bound in practice
    assert err.max() < 1e-5


def test_gemm_full_config_every_tile(g):
    """17408 x 5120 N(0, 0.015^2) weights (packed on the GPU), 2048 bf16
    tokens N(0,1) with 0.5% entries x20, seed 3.  The GEMM tiles the weights
    in 256-row tiles shared by a CTA pair (rows 0-127 of a tile on the even
    CTA, 128-255 on the odd one): two rows in each of the 68 tiles, one in
    each half, are checked for all 2048 tokens (packed bytes bit-exact,
    outputs within tolerance normwise per token over the 136 rows)."""
    import torch
    w = prefill_gemm()
    M, K = w["W"].shape
    N = w["X"].shape[0]
    Pg = g.rfp2_pack_weights(dev(w["W"]))
    rng = np.random.default_rng(3)
    rows = np.array(sorted({256 * t + h * 128 + int(rng.integers(128))
                            for t in range(M // 256) for h in range(2)}))
    rows[0], rows[-1] = 0, M - 1
    assert len(rows) == 2 * (M // 256)
    Po = rows_parallel(oracle.rfp2_pack, w["W"][rows])
    np.testing.assert_array_equal(host(Pg)[rows], Po)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = host(g.rfp2_gemm(Pg, M, K, dev(w["X"].view(np.int16)), dev_status=st))
    assert int(host(st)[0]) == 0
    ref = rows_parallel(lambda P, X: oracle.rfp2_gemm(P, P.shape[0], K, X).T, Po, w["X"]).T
    assert np.all(rel_err_rows(Y[:, rows], ref) <= TOL)
    assert np.all(np.isfinite(Y))


def test_gemm_error_codes(g):
    import torch
    P = dev(np.zeros((16, 8, 10), np.uint8))
    X = dev(np.zeros((4, 256), np.int16))
    # no workspace is needed
    assert g.rfp2_gemm_workspace_bytes(16, 256) == 0
    g.rfp2_gemm(P, 16, 256, X, workspace=torch.empty(1, dtype=torch.uint8, device="cuda"))
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemm(dev(np.zeros((12, 8, 10), np.uint8)), 12, 256, X)
    assert e.value.status == 4   # M % 16
