"""gemm_rocmfp2_mul_gb300: ROCmFP2 / HFP4G32 block-quantized GEMV and GEMM on GB300.

Thin Python binding of ``librfp2.so`` (C ABI declared in ``include/rfp2.h``).
Every function has the name of the C entry point it calls and only marshals
arguments: it takes torch CUDA tensors, allocates outputs and workspaces with
torch when the caller does not pass them, passes raw device pointers and the
current torch stream to the library, and raises :class:`RFP2Error` on a
non-zero status.  All arithmetic runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback: if the library is not built or cannot be loaded,
every call raises.

Build the library with :func:`build` (nvcc, sm_103a).
"""
from __future__ import annotations

import ctypes as C
import os
import threading

__all__ = [
    "RFP2Error", "build", "lib", "library_path", "status_str",
    "rfp2_quantize_act", "rfp2_gemv_q8", "rfp2_gemv", "rfp2_gemv_workspace_bytes",
    "rfp2_gemv_noalloc",
    "rfp2_moe_gemv", "rfp2_moe_workspace_bytes", "rfp2_gemm", "rfp2_gemm_workspace_bytes",
    "hfp4_gemv", "hfp4_gemv_workspace_bytes", "hfp4_gemm", "hfp4_gemm_workspace_bytes",
    "rfp2_nvfp4_weight_bytes", "rfp2_to_nvfp4", "rfp2_gemm_nvfp4", "rfp2_gemm_nvfp4_workspace_bytes",
    "rfp2_gemv_batched", "rfp2_gemv_batched_workspace_bytes",
    "rfp2_pack_weights", "rfp2_pack_weights_weighted", "hfp4_pack_weights", "rfp2_validate_weights",
    "rfp2_debug_half_partials", "rfp2_debug_wait_timeout", "rfp2_row_bytes", "hfp4_row_bytes",
    "rfp2_set_weight_prefetch", "rfp2_weight_prefetch",
]

MAX_BATCH = 8
_lock = threading.Lock()
_lib = None


class RFP2Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


def library_path() -> str:
    from . import buildlib as _b
    return _b.LIB


def build(force: bool = False) -> str:
    """Compile librfp2.so in-tree (nvcc, sm_103a)."""
    from . import buildlib as _b
    return _b.build(force=force)


_P, _I64, _I32, _SZ = C.c_void_p, C.c_int64, C.c_int, C.c_size_t

_SIGNATURES = {
    "rfp2_status_str": (C.c_char_p, [_I32]),
    "rfp2_version": (_I32, []),
    "rfp2_quantize_act": (_I32, [_P, _I64, _I64, _P, _P, _P]),
    "rfp2_gemv_q8": (_I32, [_P, _I64, _I64, _P, _P, _I64, _P, _P, _P]),
    "rfp2_gemv_workspace_bytes": (_SZ, [_I64, _I64]),
    "rfp2_gemv": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "rfp2_gemv_noalloc": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _P]),
    "rfp2_moe_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "rfp2_moe_gemv": (_I32, [_P, _I64, _I64, _I64, _P, _I64, _I64, _P, _P, _P, _SZ, _P, _P]),
    "rfp2_gemm_workspace_bytes": (_SZ, [_I64, _I64]),
    "rfp2_gemm": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "rfp2_gemv_batched_workspace_bytes": (_SZ, [_I64, _I64, _I64]),
    "rfp2_gemv_batched": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "hfp4_gemm_workspace_bytes": (_SZ, [_I64, _I64]),
    "hfp4_gemm": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "rfp2_nvfp4_weight_bytes": (_SZ, [_I64, _I64]),
    "rfp2_to_nvfp4": (_I32, [_P, _I64, _I64, _P, _P]),
    "rfp2_gemm_nvfp4_workspace_bytes": (_SZ, [_I64, _I64]),
    "rfp2_gemm_nvfp4": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "hfp4_gemv_workspace_bytes": (_SZ, [_I64, _I64]),
    "hfp4_gemv": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _SZ, _P, _P]),
    "rfp2_pack_weights": (_I32, [_P, _I64, _I64, _P, _P]),
    "rfp2_pack_weights_weighted": (_I32, [_P, _I64, _I64, _P, _P, _P]),
    "hfp4_pack_weights": (_I32, [_P, _I64, _I64, _P, _P, _P]),
    "rfp2_validate_weights": (_I32, [_P, _I64, _P, _P, _P]),
    "rfp2_debug_half_partials": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P]),
    "rfp2_debug_wait_timeout": (_I32, [_P, _P]),
    "rfp2_set_weight_prefetch": (_I32, [_I32]),
    "rfp2_weight_prefetch": (_I32, []),
}


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"librfp2.so is not built ({path}); run gemm_rocmfp2_mul_gb300.build()")
            L = C.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def status_str(status: int) -> str:
    try:
        return lib().rfp2_status_str(int(status)).decode()
    except Exception:
        return f"status {status}"


# -- marshalling helpers --------------------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream():
    return C.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _need(t, dtype, name, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _check(rc: int, what: str):
    if rc != 0:
        raise RFP2Error(rc, what)


def _empty(shape, dtype, like):
    return _torch().empty(shape, dtype=dtype, device=like.device)


def rfp2_row_bytes(K: int) -> int:
    """Packed bytes per ROCmFP2 row (10 bytes per 32 weights)."""
    return K // 32 * 10


def hfp4_row_bytes(K: int) -> int:
    """Bytes per HFP4G32 row (16-byte header + 17 bytes per 32 weights)."""
    return 16 + 17 * (K // 32)


def _workspace(ws, nbytes, like):
    torch = _torch()
    if ws is None:
        return torch.empty(max(nbytes, 1), dtype=torch.uint8, device=like.device)
    _need(ws, torch.uint8, "workspace")
    return ws


# -- entry points -----------------------------------------------------------------

def rfp2_quantize_act(x, q=None, d=None):
    """x fp32 [N, K] -> (q int8 [N, K], d fp32 [N, K/32])."""
    torch = _torch()
    _need(x, torch.float32, "x")
    N, K = x.shape
    q = _empty((N, K), torch.int8, x) if q is None else _need(q, torch.int8, "q")
    d = _empty((N, K // 32), torch.float32, x) if d is None else _need(d, torch.float32, "d")
    _check(lib().rfp2_quantize_act(_ptr(x), N, K, _ptr(q), _ptr(d), _stream()),
           "rfp2_quantize_act")
    return q, d


def rfp2_gemv_q8(W, M, K, q, d, y=None, dev_status=None):
    """ROCmFP2 GEMV on quantized activations: y fp32 [N, M]."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(q, torch.int8, "q")
    _need(d, torch.float32, "d")
    N = q.shape[0]
    y = _empty((N, M), torch.float32, q) if y is None else _need(y, torch.float32, "y")
    _check(lib().rfp2_gemv_q8(_ptr(W), M, K, _ptr(q), _ptr(d), N, _ptr(y), _ptr(dev_status),
                              _stream()), "rfp2_gemv_q8")
    return y


def rfp2_gemv_workspace_bytes(N: int, K: int) -> int:
    return int(lib().rfp2_gemv_workspace_bytes(N, K))


def rfp2_gemv(W, M, K, x, y=None, workspace=None, dev_status=None):
    """ROCmFP2 GEMV from fp32 activations (quantize + GEMV): y fp32 [N, M]."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(x, torch.float32, "x")
    N = x.shape[0]
    y = _empty((N, M), torch.float32, x) if y is None else _need(y, torch.float32, "y")
    nb = rfp2_gemv_workspace_bytes(N, K)
    ws = _workspace(workspace, nb, x)
    _check(lib().rfp2_gemv(_ptr(W), M, K, _ptr(x), N, _ptr(y), _ptr(ws), ws.numel(),
                           _ptr(dev_status), _stream()), "rfp2_gemv")
    return y


def rfp2_set_weight_prefetch(enable: bool) -> None:
    """Process-wide switch (default off): let the GEMV kernels start reading
    W before the kernel enqueued just before them has completed.  Turn it on
    only when no kernel that may still be running on the stream writes W."""
    _check(lib().rfp2_set_weight_prefetch(1 if enable else 0), "rfp2_set_weight_prefetch")


def rfp2_weight_prefetch() -> bool:
    """The current weight-prefetch setting."""
    return bool(lib().rfp2_weight_prefetch())


def rfp2_gemv_noalloc(W, M, K, x, y=None, dev_status=None):
    """rfp2_gemv for callers that cannot allocate device memory: the quantized
    activations go to scratch built into the library (N*K <= 65536; calls on
    one device must not overlap on the GPU).  y fp32 [N, M]; pass `y` to avoid
    the one torch allocation this wrapper would otherwise make."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(x, torch.float32, "x")
    N = x.shape[0]
    y = _empty((N, M), torch.float32, x) if y is None else _need(y, torch.float32, "y")
    _check(lib().rfp2_gemv_noalloc(_ptr(W), M, K, _ptr(x), N, _ptr(y), _ptr(dev_status),
                                   _stream()), "rfp2_gemv_noalloc")
    return y


def rfp2_moe_workspace_bytes(T: int, top_k: int, K: int) -> int:
    return int(lib().rfp2_moe_workspace_bytes(T, top_k, K))


def rfp2_moe_gemv(W, E, M, K, ids, x, y=None, workspace=None, dev_status=None):
    """MoE expert-indexed GEMV: y fp32 [T, top_k, M] = W[ids[t, j]] x_t."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(ids, torch.int32, "ids")
    _need(x, torch.float32, "x")
    T, top_k = ids.shape
    y = _empty((T, top_k, M), torch.float32, x) if y is None else _need(y, torch.float32, "y")
    ws = _workspace(workspace, rfp2_moe_workspace_bytes(T, top_k, K), x)
    _check(lib().rfp2_moe_gemv(_ptr(W), E, M, K, _ptr(ids), T, top_k, _ptr(x), _ptr(y), _ptr(ws),
                               ws.numel(), _ptr(dev_status), _stream()), "rfp2_moe_gemv")
    return y


def rfp2_gemm_workspace_bytes(M: int, K: int) -> int:
    return int(lib().rfp2_gemm_workspace_bytes(M, K))


def rfp2_gemm(W, M, K, X, Y=None, workspace=None, dev_status=None):
    """Prefill GEMM on tensor cores: Y fp32 [N, M] = X (bf16 [N, K]) W^T."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    if X.dtype == torch.bfloat16:
        X = X.view(torch.int16)
    if X.dtype not in (torch.int16, torch.uint16):
        raise TypeError("X must be bfloat16 (or its 16-bit pattern)")
    _need(X, X.dtype, "X")
    N = X.shape[0]
    Y = _empty((N, M), torch.float32, X) if Y is None else _need(Y, torch.float32, "Y")
    ws = _workspace(workspace, rfp2_gemm_workspace_bytes(M, K), X)
    _check(lib().rfp2_gemm(_ptr(W), M, K, _ptr(X), N, _ptr(Y), _ptr(ws), ws.numel(),
                           _ptr(dev_status), _stream()), "rfp2_gemm")
    return Y


def rfp2_gemv_batched_workspace_bytes(M: int, K: int, N: int) -> int:
    return int(lib().rfp2_gemv_batched_workspace_bytes(M, K, N))


def rfp2_gemv_batched(W, M, K, x, y=None, workspace=None, dev_status=None):
    """ROCmFP2 GEMV on Q8_1 activations for verify batches (tensor cores):
    y fp32 [N, M] from fp32 x [N, K]."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(x, torch.float32, "x")
    N = x.shape[0]
    y = _empty((N, M), torch.float32, x) if y is None else _need(y, torch.float32, "y")
    ws = _workspace(workspace, rfp2_gemv_batched_workspace_bytes(M, K, N), x)
    _check(lib().rfp2_gemv_batched(_ptr(W), M, K, _ptr(x), N, _ptr(y), _ptr(ws), ws.numel(),
                                   _ptr(dev_status), _stream()), "rfp2_gemv_batched")
    return y


def hfp4_gemm_workspace_bytes(M: int, K: int) -> int:
    return int(lib().hfp4_gemm_workspace_bytes(M, K))


def hfp4_gemm(W, M, K, X, Y=None, workspace=None, dev_status=None):
    """HFP4G32 prefill GEMM on tensor cores: Y fp32 [N, M] = X (bf16 [N, K]) W^T."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    if X.dtype == torch.bfloat16:
        X = X.view(torch.int16)
    if X.dtype not in (torch.int16, torch.uint16):
        raise TypeError("X must be bfloat16 (or its 16-bit pattern)")
    _need(X, X.dtype, "X")
    N = X.shape[0]
    Y = _empty((N, M), torch.float32, X) if Y is None else _need(Y, torch.float32, "Y")
    ws = _workspace(workspace, hfp4_gemm_workspace_bytes(M, K), X)
    _check(lib().hfp4_gemm(_ptr(W), M, K, _ptr(X), N, _ptr(Y), _ptr(ws), ws.numel(),
                           _ptr(dev_status), _stream()), "hfp4_gemm")
    return Y


def rfp2_nvfp4_weight_bytes(M: int, K: int) -> int:
    return int(lib().rfp2_nvfp4_weight_bytes(M, K))


def rfp2_to_nvfp4(W, M, K, out=None):
    """Exact NVFP4 image of packed ROCmFP2 weights: uint8 [rfp2_nvfp4_weight_bytes]
    (E2M1 codes [M, K/2], then scale bytes [M, K/16])."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    n = rfp2_nvfp4_weight_bytes(M, K)
    out = torch.empty(n, dtype=torch.uint8, device=W.device) if out is None else _need(out, torch.uint8, "out")
    _check(lib().rfp2_to_nvfp4(_ptr(W), M, K, _ptr(out), _stream()), "rfp2_to_nvfp4")
    return out


def rfp2_gemm_nvfp4_workspace_bytes(N: int, K: int) -> int:
    return int(lib().rfp2_gemm_nvfp4_workspace_bytes(N, K))


def rfp2_gemm_nvfp4(Wnv, M, K, X, Y=None, workspace=None, dev_status=None):
    """NVFP4 prefill GEMM on the FP4 tensor cores: Y fp32 [N, M] = NVFP4(X) Wnv^T
    (X bf16 [N, K] quantized per token into the workspace)."""
    torch = _torch()
    _need(Wnv, torch.uint8, "Wnv")
    if X.dtype == torch.bfloat16:
        X = X.view(torch.int16)
    if X.dtype not in (torch.int16, torch.uint16):
        raise TypeError("X must be bfloat16 (or its 16-bit pattern)")
    _need(X, X.dtype, "X")
    N = X.shape[0]
    Y = _empty((N, M), torch.float32, X) if Y is None else _need(Y, torch.float32, "Y")
    ws = _workspace(workspace, rfp2_gemm_nvfp4_workspace_bytes(N, K), X)
    _check(lib().rfp2_gemm_nvfp4(_ptr(Wnv), M, K, _ptr(X), N, _ptr(Y), _ptr(ws), ws.numel(),
                                 _ptr(dev_status), _stream()), "rfp2_gemm_nvfp4")
    return Y


def hfp4_gemv_workspace_bytes(N: int, K: int) -> int:
    return int(lib().hfp4_gemv_workspace_bytes(N, K))


def hfp4_gemv(W, M, K, x, y=None, workspace=None, dev_status=None):
    """HFP4G32 GEMV: y fp32 [N, M]."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(x, torch.float32, "x")
    N = x.shape[0]
    y = _empty((N, M), torch.float32, x) if y is None else _need(y, torch.float32, "y")
    ws = _workspace(workspace, hfp4_gemv_workspace_bytes(N, K), x)
    _check(lib().hfp4_gemv(_ptr(W), M, K, _ptr(x), N, _ptr(y), _ptr(ws), ws.numel(),
                           _ptr(dev_status), _stream()), "hfp4_gemv")
    return y


def rfp2_pack_weights(W, out=None):
    """fp32 W [M, K] -> ROCmFP2 blocks uint8 [M, K/32, 10] (bit-identical to the oracle)."""
    torch = _torch()
    _need(W, torch.float32, "W")
    M, K = W.shape
    out = _empty((M, K // 32, 10), torch.uint8, W) if out is None else _need(out, torch.uint8, "out")
    _check(lib().rfp2_pack_weights(_ptr(W), M, K, _ptr(out), _stream()), "rfp2_pack_weights")
    return out


def rfp2_pack_weights_weighted(W, importance, out=None):
    """fp32 W [M, K] and importance fp32 [K] -> ROCmFP2 blocks uint8 [M, K/32, 10]
    with the importance-weighted scale search."""
    torch = _torch()
    _need(W, torch.float32, "W")
    _need(importance, torch.float32, "importance")
    M, K = W.shape
    if importance.numel() != K:
        raise ValueError("importance needs one value per column")
    out = (_empty((M, K // 32, 10), torch.uint8, W) if out is None
           else _need(out, torch.uint8, "out"))
    _check(lib().rfp2_pack_weights_weighted(_ptr(W), M, K, _ptr(importance), _ptr(out),
                                            _stream()), "rfp2_pack_weights_weighted")
    return out


def hfp4_pack_weights(W, out=None, dev_status=None):
    """fp32 W [M, K] -> HFP4G32 rows uint8 [M, 16 + 17*K/32]."""
    torch = _torch()
    _need(W, torch.float32, "W")
    M, K = W.shape
    out = (_empty((M, hfp4_row_bytes(K)), torch.uint8, W) if out is None
           else _need(out, torch.uint8, "out"))
    _check(lib().hfp4_pack_weights(_ptr(W), M, K, _ptr(out), _ptr(dev_status), _stream()),
           "hfp4_pack_weights")
    return out


def rfp2_validate_weights(W, dev_status=None):
    """Count of scale bytes >= 0x7F, as a device int64 tensor of one element."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    bad = torch.zeros(1, dtype=torch.int64, device=W.device)
    _check(lib().rfp2_validate_weights(_ptr(W), W.numel() // 10, _ptr(bad), _ptr(dev_status),
                                       _stream()), "rfp2_validate_weights")
    return bad


def rfp2_debug_half_partials(W, M, K, q, partials=None):
    """int32 half sums [N, M, K/16] of the GEMV's integer path."""
    torch = _torch()
    _need(W, torch.uint8, "W")
    _need(q, torch.int8, "q")
    N = q.shape[0]
    partials = (_empty((N, M, K // 16), torch.int32, q) if partials is None
                else _need(partials, torch.int32, "partials"))
    _check(lib().rfp2_debug_half_partials(_ptr(W), M, K, _ptr(q), N, _ptr(partials), _stream()),
           "rfp2_debug_half_partials")
    return partials


def rfp2_debug_wait_timeout(dev_status):
    """Run the bounded-wait test hook: dev_status (device int32 [1]) gets
    RFP2_ETIMEOUT after the library's wait limit."""
    torch = _torch()
    _need(dev_status, torch.int32, "dev_status")
    _check(lib().rfp2_debug_wait_timeout(_ptr(dev_status), _stream()), "rfp2_debug_wait_timeout")
    return dev_status
