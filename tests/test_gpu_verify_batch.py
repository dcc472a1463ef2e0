"""GPU parity of the verify-batch ROCmFP2 GEMV (rfp2_gemv_batched: tensor
cores, weights decoded to f16 inside the GEMM kernel, activations quantized as
Q8_1 blocks and split into two f16 pieces) against the CPU oracle's int-path GEMV, through
the C ABI.  Bar: the q and d it leaves in the workspace bit-exact; outputs
within 1e-5 relative, normwise per output row (one token's [M] vector)."""
import numpy as np
import pytest

import oracle
from synth import child_rngs, decode_gemv, normal_weights
from _helpers import rel_err_rows

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


def _ws_qd(wsh, M, K, N):
    up = lambda v: (v + 255) // 256 * 256
    o = 0
    q = wsh[o:o + N * K].view(np.int8).reshape(N, K)
    o += up(N * K)
    d = wsh[o:o + N * K // 32 * 4].view(np.float32).reshape(N, K // 32)
    return q, d


@pytest.mark.parametrize("M,K,N", [
    (256, 1024, 32), (512, 4096, 128), (272, 2048, 37), (1024, 768, 200), (128, 512, 1),
    (256, 8192, 40), (144, 16384, 5),  # several read-backs of the accumulators along K
    (128, 16384, 100),  # a 128-token tile: one accumulator, eight read-backs
])
def test_verify_batch_parity(g, M, K, N):
    import torch
    r_w, r_x = child_rngs(M + K + N, 2)
    W = normal_weights(r_w, M, K, 0.02)
    x = r_x.standard_normal((N, K)).astype(np.float32)
    x[0, :64] *= 50.0  # one token with a few large blocks
    P = oracle.rfp2_pack(W)
    ws = torch.empty(g.rfp2_gemv_batched_workspace_bytes(M, K, N), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.rfp2_gemv_batched(dev(P), M, K, dev(x), workspace=ws, dev_status=st))
    assert int(host(st)[0]) == 0
    qo, do = oracle.quantize_act(x)
    qg, dg = _ws_qd(host(ws), M, K, N)
    np.testing.assert_array_equal(qg, qo)
    np.testing.assert_array_equal(dg, do)
    ref = oracle.rfp2_gemv(P, M, K, qo, do)
    err = rel_err_rows(y, ref)
    assert np.all(err <= TOL), err.max()


def test_verify_batch_matches_gemv_at_small_batch(g):
    """At a batch the dp4a GEMV also takes, both paths agree within the bar."""
    w = decode_gemv(M=2048, K=4096, N=4, seed=6)
    P = dev(oracle.rfp2_pack(w["W"]))
    x = dev(w["x"])
    y1 = host(g.rfp2_gemv(P, 2048, 4096, x))
    y2 = host(g.rfp2_gemv_batched(P, 2048, 4096, x))
    assert np.all(rel_err_rows(y2, y1) <= 2 * TOL)


@pytest.mark.parametrize("N", [32, 128])
def test_verify_batch_full_size_sampled(g, N):
    """The 14336 x 4096 decode weights (Student-t(5) x 0.02, 41 outlier columns
    x8, seed 1) packed on the GPU, N tokens N(0,1); the oracle checks 64
    sampled rows for every token."""
    import torch
    w = decode_gemv(N=4)
    M, K = w["W"].shape
    Pg = g.rfp2_pack_weights(dev(w["W"]))
    x = np.random.default_rng(N).standard_normal((N, K)).astype(np.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.rfp2_gemv_batched(Pg, M, K, dev(x), dev_status=st))
    assert int(host(st)[0]) == 0
    rows = np.sort(np.random.default_rng(N + 1).choice(M, 64, replace=False))
    Po = oracle.rfp2_pack(w["W"][rows])
    np.testing.assert_array_equal(host(Pg)[rows], Po)
    q, d = oracle.quantize_act(x)
    ref = oracle.rfp2_gemv(Po, len(rows), K, q, d)
    assert np.all(rel_err_rows(y[:, rows], ref) <= TOL)
    assert np.all(np.isfinite(y))


def test_verify_batch_errors(g):
    import torch
    P = dev(np.zeros((16, 8, 10), np.uint8))
    x = dev(np.zeros((4, 256), np.float32))
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv_batched(P, 16, 256, x, workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 9
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_gemv_batched(dev(np.zeros((12, 8, 10), np.uint8)), 12, 256, x)
    assert e.value.status == 4


@pytest.mark.parametrize("N", [3, 8])
def test_gemv_and_batched_agree_long_k(g, N):
    """At 3 and 8 tokens and K = 16384 (four accumulator read-backs along K
    on the tensor cores) both entry points meet the int path's tolerance:
    rfp2_gemv (int8 dp4a) and rfp2_gemv_batched (tensor cores)."""
    M, K = 160, 16384
    r_w, r_x = child_rngs(N + 99, 2)
    P = oracle.rfp2_pack(normal_weights(r_w, M, K, 0.02))
    x = r_x.standard_normal((N, K)).astype(np.float32)
    y = host(g.rfp2_gemv(dev(P), M, K, dev(x)))
    yb = host(g.rfp2_gemv_batched(dev(P), M, K, dev(x)))
    q, d = oracle.quantize_act(x)
    ref = oracle.rfp2_gemv(P, M, K, q, d)
    assert np.all(rel_err_rows(y, ref) <= TOL)
    assert np.all(rel_err_rows(yb, ref) <= TOL)
