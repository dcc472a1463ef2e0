"""GPU parity of the HFP4G32 GEMV (hfp4_gemv) and packer against the CPU
oracle, through the C ABI: outputs within 1e-5 relative, normwise per output
row (one token's [M] vector); packed rows bit-exact."""
import numpy as np
import pytest

import oracle
from synth import child_rngs, hfp4_gemv as hfp4_workload, normal_weights
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


def _case(g, M, K, N, seed, x=None, wscale=0.02):
    import torch
    r_w, r_x = child_rngs(seed, 2)
    W = normal_weights(r_w, M, K, wscale)
    if x is None:
        x = r_x.standard_normal((N, K)).astype(np.float32)
    P = oracle.hfp4_pack(W)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.hfp4_gemv(dev(P), M, K, dev(x), dev_status=st))
    assert int(host(st)[0]) == 0
    return y, oracle.hfp4_gemv(P, M, K, x), P, x


@pytest.mark.parametrize("M,K,N", [
    (64, 512, 1), (100, 1024, 8), (257, 2048, 3), (1000, 4096, 5), (33, 8192, 2), (16, 512, 8),
    (17, 1536, 4), (640, 8192, 1), (200, 2560, 7),
])
def test_hfp4_gemv_parity(g, M, K, N):
    y, ref, _, _ = _case(g, M, K, N, seed=M * 7 + K + N)
    err = rel_err_rows(y, ref)
    assert np.all(err <= TOL), err.max()


def test_hfp4_wide_dynamic_range_activations(g):
    """Columns of very different magnitude, and elements far below their
    column maximum (power-of-two scaling and the two-piece split)."""
    rng = np.random.default_rng(8)
    K, N, M = 2048, 6, 96
    x = rng.normal(0, 1, (N, K)) * (10.0 ** np.array([-20, -3, 0, 2, 6, 15]))[:, None]
    x[1, :64] *= 1e-6       # tiny entries next to normal ones
    x[3, 100] = 1e4         # one outlier dominating its column's scale
    y, ref, _, _ = _case(g, M, K, N, seed=9, x=x.astype(np.float32))
    assert np.all(rel_err_rows(y, ref) <= TOL)


def test_hfp4_device_packer_feeds_gemv(g):
    import torch
    M, K, N = 300, 4096, 8
    r_w, r_x = child_rngs(12, 2)
    W = (r_w.standard_t(4, (M, K)) * 0.02).astype(np.float32)
    x = r_x.standard_normal((N, K)).astype(np.float32)
    Pg = g.hfp4_pack_weights(dev(W))
    Po = oracle.hfp4_pack(W)
    np.testing.assert_array_equal(host(Pg), Po)
    y = host(g.hfp4_gemv(Pg, M, K, dev(x)))
    assert np.all(rel_err_rows(y, oracle.hfp4_gemv(Po, M, K, x)) <= TOL)


@pytest.mark.parametrize("N", [1, 8])
def test_hfp4_full_config(g, N):
    """8192 x 8192 N(0, 0.02^2) weights, seed 4, packed on the GPU: every
    packed byte of all 8192 rows bit-exact with the oracle, every output row
    within tolerance of the oracle (normwise per token over all rows)."""
    import torch
    w = hfp4_workload(N=8)
    M, K = w["W"].shape
    Pg = g.hfp4_pack_weights(dev(w["W"]))
    Po = rows_parallel(oracle.hfp4_pack, w["W"])
    np.testing.assert_array_equal(host(Pg), Po)
    x = w["x"][:N]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.hfp4_gemv(Pg, M, K, dev(x), dev_status=st))
    assert int(host(st)[0]) == 0
    ref = rows_parallel(lambda P, x: oracle.hfp4_gemv(P, P.shape[0], K, x).T, Po, x).T
    assert np.all(rel_err_rows(y, ref) <= TOL)
    assert np.all(np.isfinite(y))


def test_hfp4_block_nan_and_zero_rows(g):
    M, K, N = 48, 1024, 3
    r_w, r_x = child_rngs(5, 2)
    W = normal_weights(r_w, M, K, 0.02)
    W[7] = 0.0
    P = oracle.hfp4_pack(W)
    P[11, 16 + 17 * 5] = 0xFF   # block NaN in row 11
    x = r_x.standard_normal((N, K)).astype(np.float32)
    y = host(g.hfp4_gemv(dev(P), M, K, dev(x)))
    assert np.all(np.isnan(y[:, 11]))
    assert np.all(y[:, 7] == 0.0)
    ref = oracle.hfp4_gemv(P, M, K, x)
    keep = [m for m in range(M) if m != 11]
    assert np.all(rel_err_rows(y[:, keep], ref[:, keep]) <= TOL)


def test_hfp4_error_codes(g):
    import torch
    P = dev(np.zeros((4, 16 + 17 * 8), np.uint8))
    with pytest.raises(g.RFP2Error) as e:
        g.hfp4_gemv(P, 4, 256, dev(np.zeros((1, 256), np.float32)))
    assert e.value.status == 4   # K % 512
    P = dev(np.zeros((4, 16 + 17 * 16), np.uint8))
    with pytest.raises(g.RFP2Error) as e:
        g.hfp4_gemv(P, 4, 512, dev(np.zeros((1, 512), np.float32)),
                    workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 9
