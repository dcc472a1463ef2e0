"""rfp2_gemv_noalloc: the GEMV entry point for callers that cannot allocate
device memory (its quantized activations live in scratch built into the
library).  Called through the C ABI with buffers made before the calls, and
compared with rfp2_gemv and with the CPU oracle on two calls in a row, at
one, two, four and eight columns, with a ragged row count and with the
scratch filled to its 65536-element limit.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
from synth import child_rngs, normal_weights

pytestmark = pytest.mark.gpu
TOL = 1e-5
EWORKSPACE = 9


def _rel_rows(y, ref):
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


@pytest.mark.parametrize("M,K,N", [(1536, 4096, 4), (1001, 4096, 1), (640, 8192, 2),
                                   (512, 8192, 8)])
def test_noalloc_matches_rfp2_gemv_and_oracle_on_two_calls_in_a_row(M, K, N):
    """(512, 8192, 8) fills the scratch exactly (N*K = 65536); (1001, 4096, 1)
    has a row count that is not a multiple of any tile."""
    import torch
    import gemm_rocmfp2_mul_gb300 as g
    g.build()
    L = g.lib()
    r_w, r_x1, r_x2 = child_rngs(77 + N, 3)
    W = normal_weights(r_w, M, K, 0.02)
    P = g.rfp2_pack_weights(torch.from_numpy(W).cuda())
    xh = [r.standard_normal((N, K)).astype(np.float32) for r in (r_x1, r_x2)]
    xs = [torch.from_numpy(x).cuda() for x in xh]
    outs = [torch.empty((N, M), dtype=torch.float32, device="cuda") for _ in xs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row on the same stream, sharing the built-in scratch
    for x, y in zip(xs, outs):
        rc = L.rfp2_gemv_noalloc(C.c_void_p(P.data_ptr()), M, K, C.c_void_p(x.data_ptr()), N,
                                 C.c_void_p(y.data_ptr()), C.c_void_p(st.data_ptr()), stream)
        assert rc == 0, g.status_str(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Po = oracle.rfp2_pack(W)
    for x, xn, y in zip(xs, xh, outs):
        yh = y.cpu().numpy()
        ref = g.rfp2_gemv(P, M, K, x).cpu().numpy()
        assert np.all(_rel_rows(yh, ref) <= TOL)
        q, d = oracle.quantize_act(xn)
        assert np.all(_rel_rows(yh, oracle.rfp2_gemv(Po, M, K, q, d)) <= TOL)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import gemm_rocmfp2_mul_gb300 as g
    g.build()
    L = g.lib()
    M, K, N = 16, 40960, 2   # a supported GEMV shape with N*K = 81920 > 65536
    P = torch.zeros((M, K // 32, 10), dtype=torch.uint8, device="cuda")
    x = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    y = torch.empty((N, M), dtype=torch.float32, device="cuda")
    rc = L.rfp2_gemv_noalloc(C.c_void_p(P.data_ptr()), M, K, C.c_void_p(x.data_ptr()), N,
                             C.c_void_p(y.data_ptr()), None,
                             C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == EWORKSPACE
