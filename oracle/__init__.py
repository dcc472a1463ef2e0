"""CPU oracle for ROCmFP2 / HFP4G32 GEMV and GEMM: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
legs of ``bench.py`` may import this package.  The product library
(``gemm_rocmfp2_mul_gb300``) never imports, links or runs anything here, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``rfp2_oracle.c`` (plain single-threaded C, fp64
outputs, compiled with ``-ffp-contract=off``); this module only builds it with
gcc on first use and marshals numpy arrays through ctypes.  Each wrapper cites
the same passage as the C function it calls.

Functions whose result is not fixed by the pages (see the C file's header)
are pinned by the tests against brute force, independent library decoders,
closed forms and the pages' worked example.  The exact E2M1 tie rounding and
the scale byte chosen in exact error ties are fixed by a stated reading, not by
the pages.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rfp2_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK = 0


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no -march flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P = C.c_void_p
            I64 = C.c_int64
            sig = {
                "orc_codebook_value": (C.c_int, [C.c_int]),
                "orc_ue4m3": (C.c_int, [C.c_int, C.POINTER(C.c_double)]),
                "orc_rfp2_code": (C.c_int, [C.c_float, C.c_float]),
                "orc_rfp2_half_sse": (C.c_double, [P, C.c_int]),
                "orc_rfp2_quantize_half": (C.c_int, [P, P]),
                "orc_rfp2_pack": (C.c_int, [P, I64, I64, P]),
                "orc_rfp2_pack_weighted": (C.c_int, [P, I64, I64, P, P]),
                "orc_rfp2_half_wsse": (C.c_double, [P, P, C.c_double, C.c_int]),
                "orc_rfp2_block_sigma2": (C.c_double, [P]),
                "orc_rfp2_decode": (C.c_int, [P, I64, I64, P]),
                "orc_rfp2_count_bad_scales": (I64, [P, I64]),
                "orc_quantize_act": (C.c_int, [P, I64, I64, P, P]),
                "orc_rfp2_half_partials": (C.c_int, [P, I64, I64, P, I64, P]),
                "orc_rfp2_gemv_rows": (C.c_int, [P, I64, I64, P, I64, P, P, I64, P]),
                "orc_rfp2_gemv_brute": (C.c_int, [P, I64, I64, P, P, I64, P]),
                "orc_rfp2_moe_rows": (C.c_int, [P, I64, I64, I64, P, I64, I64, P, I64, P, P, P]),
                "orc_rfp2_gemm_rows": (C.c_int, [P, I64, I64, P, I64, P, I64, P]),
                "orc_e2m1_value": (C.c_double, [C.c_int]),
                "orc_e2m1_encode": (C.c_int, [C.c_double]),
                "orc_ue8m0": (C.c_double, [C.c_int]),
                "orc_hfp4_row_bytes": (I64, [I64]),
                "orc_hfp4_pack": (C.c_int, [P, I64, I64, P]),
                "orc_hfp4_decode": (C.c_int, [P, I64, I64, P]),
                "orc_hfp4_gemv_rows": (C.c_int, [P, I64, I64, P, I64, P, I64, P]),
                "orc_f32_to_f16_bits": (C.c_uint16, [C.c_float]),
                "orc_f16_bits_to_f32": (C.c_float, [C.c_uint16]),
                "orc_e4m3fn_value": (C.c_double, [C.c_int]),
                "orc_e4m3fn_encode": (C.c_int, [C.c_double]),
                "orc_rfp2_to_nvfp4": (C.c_int, [P, I64, I64, P, P]),
                "orc_nvfp4_quant_act": (C.c_int, [P, I64, I64, P, P, P]),
                "orc_nvfp4_gemm_rows": (C.c_int, [P, P, I64, I64, P, P, P, I64, P, I64, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _check(rc: int, what: str):
    if rc != OK:
        raise ValueError(f"oracle {what}: invalid input (rc={rc})")


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# -- ROCmFP2 -----------------------------------------------------------------

def codebook_value(code: int) -> int:
    """ROCmFP2 codebook: 00 -> -4, 01 -> -1, 10 -> +1, 11 -> +4."""
    return _load().orc_codebook_value(code)


def ue4m3(b: int) -> float:
    """UE4M3 scale byte -> scale; raises ValueError for bytes >= 0x7F."""
    s = C.c_double()
    _check(_load().orc_ue4m3(int(b), C.byref(s)), f"ue4m3({b:#x})")
    return s.value


def rfp2_code(x: float, s: float) -> int:
    """2-bit code of x at scale s (sign picks the side, |x/s| <= 2.5 inner)."""
    return _load().orc_rfp2_code(float(x), float(s))


def rfp2_half_sse(x16: np.ndarray, b: int) -> float:
    """fp64 squared reconstruction error of 16 values at scale byte b."""
    x16 = _c(x16, np.float32)
    assert x16.size == 16
    return _load().orc_rfp2_half_sse(_ptr(x16), int(b))


def rfp2_quantize_half(x16: np.ndarray) -> tuple[int, np.ndarray]:
    """Exhaustive scale search for one half: (scale byte, 16 codes)."""
    x16 = _c(x16, np.float32)
    assert x16.size == 16
    codes = np.zeros(16, np.uint8)
    b = _load().orc_rfp2_quantize_half(_ptr(x16), _ptr(codes))
    return b, codes


def rfp2_pack(W: np.ndarray) -> np.ndarray:
    """fp32 W [M, K] -> ROCmFP2 blocks uint8 [M, K/32, 10]."""
    W = _c(W, np.float32)
    M, K = W.shape
    out = np.zeros((M, K // 32, 10), np.uint8)
    _check(_load().orc_rfp2_pack(_ptr(W), M, K, _ptr(out)), "rfp2_pack")
    return out


def rfp2_pack_weighted(W: np.ndarray, importance: np.ndarray) -> np.ndarray:
    """fp32 W [M, K] and importance fp32 [K] -> uint8 [M, K/32, 10] with the
    importance-weighted scale search (same block, codebook and code rule)."""
    W = _c(W, np.float32)
    imp = _c(importance, np.float32).reshape(-1)
    M, K = W.shape
    if imp.size != K:
        raise ValueError("importance needs one value per column")
    out = np.zeros((M, K // 32, 10), np.uint8)
    _check(_load().orc_rfp2_pack_weighted(_ptr(W), M, K, _ptr(imp), _ptr(out)),
           "rfp2_pack_weighted")
    return out


def rfp2_half_wsse(x16: np.ndarray, imp16: np.ndarray, sigma2: float, b: int) -> float:
    """Weighted squared error of one 16-value half at scale byte b."""
    return float(_load().orc_rfp2_half_wsse(_ptr(_c(x16, np.float32)), _ptr(_c(imp16, np.float32)),
                                            float(sigma2), int(b)))


def rfp2_block_sigma2(x32: np.ndarray) -> float:
    """sigma^2 of the weighted objective: twice the mean of x^2 over the block."""
    return float(_load().orc_rfp2_block_sigma2(_ptr(_c(x32, np.float32))))


def rfp2_decode(P: np.ndarray, M: int, K: int) -> np.ndarray:
    """Packed blocks -> reconstructed fp32 weights [M, K]."""
    P = _c(P, np.uint8)
    assert P.size == M * K // 32 * 10
    out = np.zeros((M, K), np.float32)
    _check(_load().orc_rfp2_decode(_ptr(P), M, K, _ptr(out)), "rfp2_decode")
    return out


def rfp2_count_bad_scales(P: np.ndarray) -> int:
    """Number of scale bytes >= 0x7F in a packed buffer."""
    P = _c(P, np.uint8)
    return int(_load().orc_rfp2_count_bad_scales(_ptr(P), P.size // 10))


def quantize_act(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 x [N, K] -> (q int8 [N, K], d fp32 [N, K/32])."""
    x = _c(np.atleast_2d(x), np.float32)
    N, K = x.shape
    q = np.zeros((N, K), np.int8)
    d = np.zeros((N, K // 32), np.float32)
    _check(_load().orc_quantize_act(_ptr(x), N, K, _ptr(q), _ptr(d)), "quantize_act")
    return q, d


def rfp2_half_partials(P: np.ndarray, M: int, K: int, q: np.ndarray) -> np.ndarray:
    """int32 half sums [N, M, K/16]."""
    P = _c(P, np.uint8)
    q = _c(np.atleast_2d(q), np.int8)
    N = q.shape[0]
    out = np.zeros((N, M, K // 16), np.int32)
    _check(_load().orc_rfp2_half_partials(_ptr(P), M, K, _ptr(q), N, _ptr(out)), "half_partials")
    return out


def rfp2_gemv(P: np.ndarray, M: int, K: int, q: np.ndarray, d: np.ndarray,
              rows=None) -> np.ndarray:
    """fp64 y [N, len(rows)] = sum_blocks dA*(d0*S0 + d1*S1) (int path)."""
    P = _c(P, np.uint8)
    q = _c(np.atleast_2d(q), np.int8)
    d = _c(np.atleast_2d(d), np.float32)
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    N = q.shape[0]
    y = np.zeros((N, rows.size), np.float64)
    _check(_load().orc_rfp2_gemv_rows(_ptr(P), M, K, _ptr(rows), rows.size, _ptr(q), _ptr(d),
                                      N, _ptr(y)), "rfp2_gemv")
    return y


def rfp2_gemv_brute(P: np.ndarray, M: int, K: int, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    """fp64 y [N, M] = sum_k w_k * (q_k * dA), one weight at a time."""
    P = _c(P, np.uint8)
    q = _c(np.atleast_2d(q), np.int8)
    d = _c(np.atleast_2d(d), np.float32)
    N = q.shape[0]
    y = np.zeros((N, M), np.float64)
    _check(_load().orc_rfp2_gemv_brute(_ptr(P), M, K, _ptr(q), _ptr(d), N, _ptr(y)), "gemv_brute")
    return y


def rfp2_moe(P: np.ndarray, E: int, M: int, K: int, ids: np.ndarray, q: np.ndarray,
             d: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y [T, top_k, len(rows)]: row r of expert ids[t, j] times token t."""
    P = _c(P, np.uint8)
    ids = _c(ids, np.int32)
    q = _c(q, np.int8)
    d = _c(d, np.float32)
    T, top_k = ids.shape
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((T, top_k, rows.size), np.float64)
    _check(_load().orc_rfp2_moe_rows(_ptr(P), E, M, K, _ptr(ids), T, top_k, _ptr(rows), rows.size,
                                     _ptr(q), _ptr(d), _ptr(y)), "rfp2_moe")
    return y


def rfp2_gemm(P: np.ndarray, M: int, K: int, X_bf16: np.ndarray, rows=None) -> np.ndarray:
    """fp64 Y [N, len(rows)] = X (bf16 bits [N, K]) times decoded weight rows."""
    P = _c(P, np.uint8)
    X = _c(X_bf16, np.uint16)
    N = X.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((N, rows.size), np.float64)
    _check(_load().orc_rfp2_gemm_rows(_ptr(P), M, K, _ptr(X), N, _ptr(rows), rows.size, _ptr(y)),
           "rfp2_gemm")
    return y


# -- HFP4G32 -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().orc_e2m1_value(int(code))


def e2m1_encode(v: float) -> int:
    return _load().orc_e2m1_encode(float(v))


def ue8m0(e: int) -> float:
    return _load().orc_ue8m0(int(e))


def hfp4_row_bytes(K: int) -> int:
    return int(_load().orc_hfp4_row_bytes(K))


def hfp4_pack(W: np.ndarray) -> np.ndarray:
    """fp32 W [M, K] -> HFP4G32 rows uint8 [M, 16 + 17*K/32]."""
    W = _c(W, np.float32)
    M, K = W.shape
    out = np.zeros((M, hfp4_row_bytes(K)), np.uint8)
    _check(_load().orc_hfp4_pack(_ptr(W), M, K, _ptr(out)), "hfp4_pack")
    return out


def hfp4_decode(P: np.ndarray, M: int, K: int) -> np.ndarray:
    """HFP4G32 rows -> fp64 weights [M, K] (NaN for block byte 0xFF)."""
    P = _c(P, np.uint8)
    out = np.zeros((M, K), np.float64)
    _check(_load().orc_hfp4_decode(_ptr(P), M, K, _ptr(out)), "hfp4_decode")
    return out


def hfp4_gemv(P: np.ndarray, M: int, K: int, x: np.ndarray, rows=None) -> np.ndarray:
    """fp64 y [N, len(rows)] = sum_b rs*2^(e-127) * sum_i lut[c_i] * x_i."""
    P = _c(P, np.uint8)
    x = _c(np.atleast_2d(x), np.float32)
    N = x.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((N, rows.size), np.float64)
    _check(_load().orc_hfp4_gemv_rows(_ptr(P), M, K, _ptr(rows), rows.size, _ptr(x), N, _ptr(y)),
           "hfp4_gemv")
    return y


def hfp4_gemm(P: np.ndarray, M: int, K: int, X_bf16: np.ndarray, rows=None) -> np.ndarray:
    """Prefill: fp64 Y [N, len(rows)] = sum_k w[m, k] * X[n, k] for bf16 tokens
    X (given as 16-bit patterns): the GEMV loop formula of hfp4_gemv over every
    token, each bf16 value widened exactly to fp32 (no activation
    quantization on this path)."""
    X = np.ascontiguousarray(np.atleast_2d(X_bf16)).view(np.uint16)
    x = (X.astype(np.uint32) << 16).view(np.float32)
    return hfp4_gemv(P, M, K, x, rows)


def f32_to_f16_bits(v: float) -> int:
    return int(_load().orc_f32_to_f16_bits(float(v)))


def f16_bits_to_f32(b: int) -> float:
    return float(_load().orc_f16_bits_to_f32(int(b)))


# -- Block-scaled FP4 (NVFP4) form ---------------------------------------------

def e4m3fn_value(b: int) -> float:
    return float(_load().orc_e4m3fn_value(int(b)))


def e4m3fn_encode(v: float) -> int:
    return int(_load().orc_e4m3fn_encode(float(v)))


def rfp2_to_nvfp4(P: np.ndarray, M: int, K: int):
    """ROCmFP2 blocks -> exact NVFP4 weights: E2M1 codes uint8 [M, K] (one per
    byte) and E4M3FN scale bytes uint8 [M, K/16]."""
    P = _c(P, np.uint8)
    codes = np.zeros((M, K), np.uint8)
    sb = np.zeros((M, K // 16), np.uint8)
    _check(_load().orc_rfp2_to_nvfp4(_ptr(P), M, K, _ptr(codes), _ptr(sb)), "rfp2_to_nvfp4")
    return codes, sb


def nvfp4_quant_act(x: np.ndarray):
    """fp32 x [N, K] -> (E2M1 codes uint8 [N, K], scale bytes uint8 [N, K/16],
    global factors g fp32 [N]); value = E2M1 * E4M3FN(byte) / g."""
    x = _c(np.atleast_2d(x), np.float32)
    N, K = x.shape
    codes = np.zeros((N, K), np.uint8)
    sb = np.zeros((N, K // 16), np.uint8)
    g = np.zeros(N, np.float32)
    _check(_load().orc_nvfp4_quant_act(_ptr(x), N, K, _ptr(codes), _ptr(sb), _ptr(g)),
           "nvfp4_quant_act")
    return codes, sb, g


def nvfp4_gemm(wc, ws, M: int, K: int, xc, xs, g, rows=None) -> np.ndarray:
    """fp64 y [N, len(rows)] = (1/g_n) sum_k wval[m, k] * xval[n, k] with both
    operands in NVFP4 form."""
    wc, ws, xc, xs = (_c(a, np.uint8) for a in (wc, ws, xc, xs))
    g = _c(g, np.float32)
    N = xc.shape[0]
    rows = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    y = np.zeros((N, rows.size), np.float64)
    _check(_load().orc_nvfp4_gemm_rows(_ptr(wc), _ptr(ws), M, K, _ptr(xc), _ptr(xs), _ptr(g), N,
                                       _ptr(rows), rows.size, _ptr(y)), "nvfp4_gemm")
    return y
