"""GPU parity of the block-scaled FP4 (NVFP4) prefill GEMM against the CPU
oracle, through the C ABI.

- The NVFP4 weight image (rfp2_to_nvfp4) is bit-exact: E2M1 codes and scale
  bytes ("ROCmFP2 codebook research report", 02 Quantization: codebook * s(b)
  = (codebook / 2) * E4M3FN(b)).
- The per-token activation quantization (codes, scale bytes, g), read back
  from the workspace, is bit-exact with oracle.nvfp4_quant_act.
- Y is within 1e-5 relative, normwise per token row, of oracle.nvfp4_gemm on
  those operands: every product is exact, only the fp32 accumulation inside
  the tensor cores differs from the fp64 sum.
"""
import numpy as np
import pytest

import oracle
from synth import child_rngs, float32_to_bf16_bits, normal_weights, outlier_bf16_activations, prefill_gemm
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


def unpack_nibbles(b):
    b = np.asarray(b, np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), np.uint8)
    out[..., 0::2] = b & 15
    out[..., 1::2] = b >> 4
    return out


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def tokens(kind, rng, N, K):
    if kind == "normal":
        return float32_to_bf16_bits(rng.standard_normal((N, K)).astype(np.float32))
    if kind == "outliers":
        return outlier_bf16_activations(rng, N, K)
    if kind == "wide":  # blocks far below the row maximum: small and subnormal scales
        x = rng.standard_normal((N, K)).astype(np.float32)
        x *= np.float32(2.0) ** rng.integers(-40, 1, (N, K // 16)).repeat(16, axis=1).astype(np.float32)
        return float32_to_bf16_bits(x)
    if kind == "zeros":  # an all-zero row, zero blocks, and signed zeros
        x = rng.standard_normal((N, K)).astype(np.float32)
        x[0] = 0.0
        x[1, :64] = 0.0
        x[1, 64:80] = -0.0
        return float32_to_bf16_bits(x)
    raise ValueError(kind)


def run(g, P, M, K, Xbits):
    import torch
    N = Xbits.shape[0]
    Wnv = g.rfp2_to_nvfp4(dev(P), M, K)
    ws = torch.empty(g.rfp2_gemm_nvfp4_workspace_bytes(N, K), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Y = g.rfp2_gemm_nvfp4(Wnv, M, K, dev(Xbits.view(np.int16)), workspace=ws, dev_status=st)
    assert int(host(st)[0]) == 0
    return host(Y), host(Wnv), host(ws)


def split_workspace(ws, N, K):
    up = lambda v: (v + 255) // 256 * 256
    codes = unpack_nibbles(ws[:N * K // 2].reshape(N, K // 2))
    o = up(N * K // 2)
    sb = ws[o:o + N * K // 16].reshape(N, K // 16)
    o += up(N * K // 16)
    gg = ws[o:o + 4 * N].view(np.float32)
    return codes, sb, gg


def test_weight_image_bit_exact(g):
    M, K = 96, 1024
    P = oracle.rfp2_pack(normal_weights(child_rngs(1, 1)[0], M, K, 0.02))
    img = host(g.rfp2_to_nvfp4(dev(P), M, K))
    assert img.size == g.rfp2_nvfp4_weight_bytes(M, K)
    wc, ws = oracle.rfp2_to_nvfp4(P, M, K)
    np.testing.assert_array_equal(unpack_nibbles(img[:M * K // 2].reshape(M, K // 2)), wc)
    np.testing.assert_array_equal(img[M * K // 2:].reshape(M, K // 16), ws)


@pytest.mark.parametrize("kind", ["normal", "outliers", "wide", "zeros"])
def test_activation_quantization_bit_exact(g, kind):
    M, K, N = 128, 2048, 37
    rng = np.random.default_rng(len(kind))
    P = oracle.rfp2_pack(normal_weights(child_rngs(2, 1)[0], M, K, 0.02))
    X = tokens(kind, rng, N, K)
    _, _, ws = run(g, P, M, K, X)
    codes, sb, gg = split_workspace(ws, N, K)
    rc, rs, rg = oracle.nvfp4_quant_act(bf16_to_f32(X))
    np.testing.assert_array_equal(gg, rg)
    np.testing.assert_array_equal(sb, rs)
    np.testing.assert_array_equal(codes, rc)


@pytest.mark.parametrize("M,K,N,kind", [
    (128, 256, 128, "normal"), (256, 512, 37, "outliers"), (200, 1024, 130, "wide"),
    (1000, 2048, 300, "normal"), (384, 5120, 64, "outliers"), (130, 768, 257, "zeros"),
])
def test_gemm_parity(g, M, K, N, kind):
    """Ragged row tiles (M % 128) and token tiles (N % 128), several K."""
    rng = np.random.default_rng(M + N)
    P = oracle.rfp2_pack(normal_weights(child_rngs(M + K, 1)[0], M, K, 0.015))
    X = tokens(kind, rng, N, K)
    Y, img, ws = run(g, P, M, K, X)
    xc, xs, gg = oracle.nvfp4_quant_act(bf16_to_f32(X))
    wc, wsb = oracle.rfp2_to_nvfp4(P, M, K)
    rows = np.arange(M, dtype=np.int64)
    ref = rows_parallel(lambda r: oracle.nvfp4_gemm(wc, wsb, M, K, xc, xs, gg, rows=r).T, rows).T
    err = rel_err_rows(Y, ref)
    assert np.all(err <= TOL), err.max()
    if kind == "zeros":
        assert np.all(Y[0] == 0.0)


def test_gemm_full_config_sampled(g):
    """The prefill workload (ROCmFP2 [17408, 5120], 2048 bf16 tokens with
    0.5 % x20 outliers, seed 3): one weight row in each of the 136 row tiles
    (a different position in each), every token; the whole workspace
    quantization of all 2048 tokens bit-exact."""
    import torch
    w = prefill_gemm()
    M, K = w["W"].shape
    N = w["X"].shape[0]
    Pd = g.rfp2_pack_weights(torch.from_numpy(w["W"]).cuda())
    Y, img, ws = run(g, host(Pd), M, K, w["X"])
    codes, sb, gg = split_workspace(ws, N, K)
    xc, xs, rg = oracle.nvfp4_quant_act(bf16_to_f32(w["X"]))
    np.testing.assert_array_equal(gg, rg)
    np.testing.assert_array_equal(sb, xs)
    np.testing.assert_array_equal(codes, xc)
    rows = np.array([128 * t + (37 * t) % 128 for t in range(M // 128)], np.int64)
    wc = unpack_nibbles(img[:M * K // 2].reshape(M, K // 2))[rows]
    wsb = img[M * K // 2:].reshape(M, K // 16)[rows]
    Pr = host(Pd)[rows]
    owc, ows = oracle.rfp2_to_nvfp4(Pr, rows.size, K)
    np.testing.assert_array_equal(wc, owc)
    np.testing.assert_array_equal(wsb, ows)
    sel = np.arange(rows.size, dtype=np.int64)
    ref = rows_parallel(lambda r: oracle.nvfp4_gemm(owc, ows, rows.size, K, xc, xs, rg, rows=r).T, sel).T
    err = rel_err_rows(Y[:, rows], ref)
    assert np.all(err <= TOL), err.max()


def test_gemm_single_token_and_zero_weights(g):
    """N = 1 (a 128-token tile with 127 zero-filled rows) and an all-zero
    weight row (scale byte 0, codes +-0.5 times 0) give exact zeros there."""
    M, K = 256, 1024
    W = normal_weights(child_rngs(5, 1)[0], M, K, 0.02)
    W[3] = 0.0
    P = oracle.rfp2_pack(W)
    X = float32_to_bf16_bits(np.random.default_rng(9).standard_normal((1, K)).astype(np.float32))
    Y, img, ws = run(g, P, M, K, X)
    xc, xs, gg = oracle.nvfp4_quant_act(bf16_to_f32(X))
    wc, wsb = oracle.rfp2_to_nvfp4(P, M, K)
    ref = oracle.nvfp4_gemm(wc, wsb, M, K, xc, xs, gg)
    assert np.all(rel_err_rows(Y, ref) <= TOL)
    assert Y[0, 3] == 0.0


def test_error_codes(g):
    import ctypes as C
    import torch
    L = g.lib()
    OK, EINVAL, ESHAPE, EALIGN, EUNSUPPORTED, EWORKSPACE = 0, 1, 2, 3, 4, 9
    p = C.c_void_p
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    b = p(buf.data_ptr())
    s = p(torch.cuda.current_stream().cuda_stream)
    assert L.rfp2_to_nvfp4(None, 4, 64, b, s) == EINVAL
    assert L.rfp2_to_nvfp4(b, 4, 40, b, s) == ESHAPE
    assert L.rfp2_to_nvfp4(b, 4, 64, p(buf.data_ptr() + 8), s) == EALIGN
    assert L.rfp2_nvfp4_weight_bytes(4, 64) == 4 * 32 + 4 * 4
    assert L.rfp2_gemm_nvfp4(None, 128, 256, b, 1, b, b, 1 << 20, None, s) == EINVAL
    assert L.rfp2_gemm_nvfp4(b, 128, 256, b, 0, b, b, 1 << 20, None, s) == ESHAPE
    assert L.rfp2_gemm_nvfp4(b, 128, 384, b, 1, b, b, 1 << 20, None, s) == EUNSUPPORTED
    assert L.rfp2_gemm_nvfp4(b, 128, 256, b, 1, b, b, 16, None, s) == EWORKSPACE
    assert L.rfp2_gemm_nvfp4(b, 128, 256, p(buf.data_ptr() + 8), 1, b, b, 1 << 20, None, s) == EALIGN
    torch.cuda.synchronize()
