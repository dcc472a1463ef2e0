"""Shared helpers for the tests: golden-file parsing and independent decoders.

The decoders here are written against independent references (torch's
float8_e4m3fn / float8_e8m0fnu dtypes, numpy's float16) so that they pin the
oracle instead of repeating it.
"""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str) -> dict:
    """Parse a 'key value...' fixture; '#' lines are comments (citations)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            conv = []
            for v in vals:
                conv.append(int(v, 16) if v.startswith("0x") else float(v))
            out[key] = conv[0] if len(conv) == 1 else conv
    return out


def e4m3fn_half_table() -> np.ndarray:
    """float64 [256]: torch's OCP E4M3FN decode of every byte, halved."""
    import torch
    b = torch.arange(256, dtype=torch.uint8)
    return (b.view(torch.float8_e4m3fn).to(torch.float64) / 2).numpy()


def unpack_codes(P: np.ndarray, M: int, K: int) -> np.ndarray:
    """uint8 codes [M, K] from packed blocks: byte i//4 of a block, bits 2*(i%4)."""
    P = np.asarray(P, np.uint8).reshape(M, K // 32, 10)
    i = np.arange(32)
    byte = P[:, :, i // 4]
    return ((byte >> (2 * (i % 4))) & 3).reshape(M, K).astype(np.uint8)


def decode_weights_independent(P: np.ndarray, M: int, K: int) -> np.ndarray:
    """float64 [M, K]: levels [-4,-1,1,4][code] times E4M3FN(scale byte)/2."""
    P = np.asarray(P, np.uint8).reshape(M, K // 32, 10)
    levels = np.array([-4.0, -1.0, 1.0, 4.0])
    table = e4m3fn_half_table()
    scales = table[P[:, :, 8:10]]                      # [M, nb, 2]
    s = np.repeat(scales, 16, axis=2).reshape(M, K)     # per weight
    return levels[unpack_codes(P, M, K)] * s


# OCP MX v1.0 E2M1 magnitudes by the low three code bits (bit 3 is the sign).
E2M1_OCP = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def decode_hfp4_independent(P: np.ndarray, M: int, K: int, row_scale: bool = True) -> np.ndarray:
    """float64 [M, K] from HFP4G32 rows, with numpy alone: row_scale_a as the
    little-endian f16 in bytes 0-1, then per 17-byte block the UE8M0 byte
    (2^(e-127), 0xFF -> NaN) and 16 code bytes, the low nibble the even
    element.  row_scale=False leaves out row_scale_a."""
    P = np.asarray(P, np.uint8).reshape(M, -1)
    nb = K // 32
    rs = P[:, 0:2].copy().view("<f2").astype(np.float64).reshape(M)
    blocks = P[:, 16:16 + 17 * nb].reshape(M, nb, 17)
    e = blocks[:, :, 0].astype(np.int64)
    scale = np.where(e == 255, np.nan, np.ldexp(1.0, e - 127))
    codes = blocks[:, :, 1:]
    c = np.stack([codes & 15, codes >> 4], axis=-1).reshape(M, nb, 32)
    val = np.where(c & 8, -1.0, 1.0) * E2M1_OCP[c & 7] * scale[:, :, None]
    if row_scale:
        val = val * rs[:, None, None]
    return val.reshape(M, K)


def bf16_bits_to_f64(X: np.ndarray) -> np.ndarray:
    X = np.ascontiguousarray(X).view(np.uint16)
    return (X.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def rel_err_rows(y, ref) -> np.ndarray:
    """Normwise relative error per row: ||y - ref||_2 / ||ref||_2."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.linalg.norm(y - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    return num / np.where(den == 0, 1.0, den)


def oracle_threads() -> int:
    import os
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def rows_parallel(fn, W, *args, threads=None):
    """fn(W[rows], *args) over contiguous row ranges on host threads (the
    oracle's ctypes calls release the GIL), concatenated along axis 0."""
    from concurrent.futures import ThreadPoolExecutor
    W = np.ascontiguousarray(W)
    n = W.shape[0]
    t = min(threads or oracle_threads(), max(1, n))
    cuts = [n * i // t for i in range(t + 1)]
    with ThreadPoolExecutor(t) as ex:
        parts = list(ex.map(lambda i: fn(np.ascontiguousarray(W[cuts[i]:cuts[i + 1]]), *args),
                            range(t)))
    return np.concatenate(parts, axis=0)
