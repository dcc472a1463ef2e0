"""GPU parity of the MoE expert-indexed GEMV (rfp2_moe_gemv) against the
CPU oracle, through the C ABI: y[t, j, :] = W[ids[t, j]] x_t, within 1e-5
relative normwise per output row; ids outside [0, E) give NaN rows and
RFP2_EBADID without touching memory."""
import numpy as np
import pytest

import oracle
from synth import child_rngs, moe_expert_weights, moe_gemv, routing_ids
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


def _run(g, P, E, M, K, ids, x):
    import torch
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.rfp2_moe_gemv(dev(P), E, M, K, dev(ids), dev(x), dev_status=st))
    return y, int(host(st)[0])


def _oracle(P, E, M, K, ids, x):
    q, d = oracle.quantize_act(x)
    return oracle.rfp2_moe(P, E, M, K, ids, q, d)


@pytest.mark.parametrize("E,M,K,T,top_k", [
    (8, 64, 512, 5, 3), (16, 200, 2048, 16, 8), (4, 96, 4096, 3, 2), (32, 130, 256, 7, 4),
    (3, 512, 1024, 12, 1),
])
def test_moe_parity(g, E, M, K, T, top_k):
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=E + M)
    P = np.stack([oracle.rfp2_pack(w["W"][e]) for e in range(E)])
    y, st = _run(g, P, E, M, K, w["ids"], w["x"])
    assert st == 0
    ref = _oracle(P, E, M, K, w["ids"], w["x"])
    err = rel_err_rows(y.reshape(T * top_k, M), ref.reshape(T * top_k, M))
    assert np.all(err <= TOL), err.max()


def test_moe_crowded_expert_and_duplicates(g):
    """Many tokens on one expert (groups of 4 split), a token routed twice to
    the same expert, and unused experts."""
    E, M, K, T, top_k = 6, 80, 512, 11, 3
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=3)
    ids = w["ids"].copy()
    ids[:, 0] = 2          # expert 2 gets every token
    ids[4, 1] = ids[4, 2] = 5
    P = np.stack([oracle.rfp2_pack(w["W"][e]) for e in range(E)])
    y, st = _run(g, P, E, M, K, ids, w["x"])
    assert st == 0
    ref = _oracle(P, E, M, K, ids, w["x"])
    assert np.all(rel_err_rows(y.reshape(-1, M), ref.reshape(-1, M)) <= TOL)


def test_moe_bad_ids_give_nan_rows_and_status(g):
    E, M, K, T, top_k = 5, 64, 256, 4, 2
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=4)
    ids = w["ids"].copy()
    ids[1, 0] = E
    ids[3, 1] = -7
    ids[2, 1] = 0x7FFFFFFF
    P = np.stack([oracle.rfp2_pack(w["W"][e]) for e in range(E)])
    y, st = _run(g, P, E, M, K, ids, w["x"])
    assert st == 7   # RFP2_EBADID
    bad = [(1, 0), (3, 1), (2, 1)]
    for t, j in bad:
        assert np.all(np.isnan(y[t, j]))
    good = np.ones((T, top_k), bool)
    for t, j in bad:
        good[t, j] = False
    ok_ids = np.where(good, ids, 0)
    ref = _oracle(P, E, M, K, ok_ids, w["x"])
    assert np.all(rel_err_rows(y[good], ref[good]) <= TOL)


def test_moe_full_config(g):
    """256 experts of 768 x 2048 Student-t(5)*0.02 weights (packed on the GPU),
    16 tokens, top-8 distinct experts per token, seed 2; every row of every
    touched expert is packed by the oracle and checked bit-exactly, and every
    (token, slot) output row is checked against the oracle over all 768 rows."""
    import torch
    E, M, K, T, top_k = 256, 768, 2048, 16, 8
    w = moe_gemv(E=E, M=M, K=K, T=T, top_k=top_k, seed=2, experts=False)
    ids = w["ids"]
    Pg = torch.empty((E, M, K // 32, 10), dtype=torch.uint8, device="cuda")
    touched = sorted(set(ids.ravel().tolist()))
    for e in range(E):
        We = dev(moe_expert_weights(2, E, M, K, e))
        g.rfp2_pack_weights(We, out=Pg[e])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = host(g.rfp2_moe_gemv(Pg, E, M, K, dev(ids), dev(w["x"]), dev_status=st))
    assert int(host(st)[0]) == 0
    q, d = oracle.quantize_act(w["x"])
    Pgh = host(Pg)
    Wt = np.concatenate([moe_expert_weights(2, E, M, K, e) for e in touched])
    Po_all = rows_parallel(oracle.rfp2_pack, Wt).reshape(len(touched), M, K // 32, 10)
    for i, e in enumerate(touched):
        np.testing.assert_array_equal(Pgh[e], Po_all[i])
        for t, j in zip(*np.nonzero(ids == e)):
            ref = oracle.rfp2_gemv(Po_all[i], M, K, q[t:t + 1], d[t:t + 1])
            assert rel_err_rows(y[t, j][None], ref)[0] <= TOL
    assert np.all(np.isfinite(y))


def test_moe_error_codes(g):
    import torch
    P = dev(np.zeros((2, 16, 8, 10), np.uint8))
    ids = dev(np.zeros((2, 2), np.int32))
    x = dev(np.zeros((2, 256), np.float32))
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_moe_gemv(P, 2, 16, 256, ids, x, workspace=torch.empty(8, dtype=torch.uint8,
                                                                    device="cuda"))
    assert e.value.status == 9
    with pytest.raises(g.RFP2Error) as e:
        g.rfp2_moe_gemv(dev(np.zeros((2, 16, 3, 10), np.uint8)), 2, 16, 96,
                        ids, dev(np.zeros((2, 96), np.float32)))
    assert e.value.status == 4
