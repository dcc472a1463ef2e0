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


def rel_err_rows(y, ref) -> np.ndarray:
    """Normwise relative error per row: ||y - ref||_2 / ||ref||_2."""
    y = np.asarray(y, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.linalg.norm(y - ref, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    return num / np.where(den == 0, 1.0, den)
