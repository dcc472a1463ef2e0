"""rfp2_gemv_noalloc: the GEMV entry point for callers that cannot allocate
device memory (its quantized activations live in scratch built into the
library).  Called through the C ABI with buffers made before the calls, and
compared with rfp2_gemv on two calls in a row.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest

from synth import child_rngs, normal_weights

pytestmark = pytest.mark.gpu
TOL = 1e-5
EWORKSPACE = 9


def _rel_rows(y, ref):
    y = y.astype(np.float64)
    ref = ref.astype(np.float64)
    return np.linalg.norm(y - ref, axis=1) / np.linalg.norm(ref, axis=1)


def test_noalloc_matches_rfp2_gemv_on_two_calls_in_a_row():
    import torch
    import gemm_rocmfp2_mul_gb300 as g
    g.build()
    L = g.lib()
    M, K, N = 1536, 4096, 4
    r_w, r_x1, r_x2 = child_rngs(77, 3)
    Wd = torch.from_numpy(normal_weights(r_w, M, K, 0.02)).cuda()
    P = g.rfp2_pack_weights(Wd)
    xs = [torch.from_numpy(r.standard_normal((N, K)).astype(np.float32)).cuda()
          for r in (r_x1, r_x2)]
    outs = [torch.empty((N, M), dtype=torch.float32, device="cuda") for _ in xs]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row on the same stream, sharing the built-in scratch
    for x, y in zip(xs, outs):
        rc = L.rfp2_gemv_noalloc(C.c_void_p(P.data_ptr()), M, K, C.c_void_p(x.data_ptr()), N,
                                 C.c_void_p(y.data_ptr()), C.c_void_p(st.data_ptr()), stream)
        assert rc == 0, g.status_str(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for x, y in zip(xs, outs):
        ref = g.rfp2_gemv(P, M, K, x).cpu().numpy()
        assert np.all(_rel_rows(y.cpu().numpy(), ref) <= TOL)


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
