"""Python binding of libparallax.so (Parallax attention on B300, sm_103a).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  The C entry points and
their contracts are declared in ``include/parallax.h``; the functions here have
the same names and take torch tensors instead of raw pointers.

If the shared library has not been built, importing succeeds but every call
raises ``PlxLibraryMissing``; there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PLX_OK", "PLX_ERR_INVALID_ARG", "PLX_ERR_UNSUPPORTED", "PLX_ERR_CUDA", "PLX_ERR_TIMEOUT",
    "PLX_ERR_TOO_LARGE", "parallax_fwd_noalloc", "parallax_step_host",
    "PLX_FP32", "PLX_BF16", "PLX_PATH_AUTO", "PLX_PATH_SIMT", "PLX_PATH_TC",
    "PlxError", "PlxLibraryMissing", "lib", "lib_path", "exported_symbols",
    "parallax_fwd", "parallax_fwd_ws", "parallax_bwd", "parallax_fwd_workspace_bytes",
    "parallax_bwd_workspace_bytes", "parallax_last_device_error", "parallax_set_path",
    "parallax_strerror", "parallax_launch_count", "parallax_timing_enable", "parallax_timing_collect",
    "parallax_timing_get", "parallax_timing_reset", "kernel_times",
    "parallax_fwd_bwd", "parallax_fwd_bwd_workspace_bytes",
    "parallax_decode", "parallax_decode_workspace_bytes", "parallax_decode_probe",
    "parallax_decode_probe_workspace_bytes",
    "parallax_fwd_probe", "parallax_fwd_probe_workspace_bytes", "parallax_set_wait_limit",
    "parallax_set_persistent_ctas",
]

PLX_OK, PLX_ERR_INVALID_ARG, PLX_ERR_UNSUPPORTED, PLX_ERR_CUDA, PLX_ERR_TIMEOUT = 0, 1, 2, 3, 4
PLX_ERR_TOO_LARGE = 5
PLX_FP32, PLX_BF16 = 0, 1
PLX_PATH_AUTO, PLX_PATH_SIMT, PLX_PATH_TC = 0, 1, 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libparallax.so")
_lib = None

# Every symbol include/parallax.h declares, with its ctypes signature.
_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "parallax_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_bwd": (_i, [_vp] * 12 + [_i, _i, _i, _i, _i, _vp]),
    "parallax_last_device_error": (_i, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "parallax_set_path": (_i, [_i]),
    "parallax_set_persistent_ctas": (_i, [_i]),
    "parallax_set_wait_limit": (_i, [ctypes.c_longlong]),
    "parallax_strerror": (ctypes.c_char_p, [_i]),
    "parallax_launch_count": (ctypes.c_ulonglong, []),
    "parallax_timing_enable": (_i, [_i]),
    "parallax_timing_collect": (_i, []),
    "parallax_timing_get": (_i, [_i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_longlong)]),
    "parallax_timing_reset": (None, []),
    "parallax_decode": (_i, [_vp] * 8 + [_i, _i, _i, _i, _i, _vp]),
    "parallax_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_decode_probe": (_i, [_vp] * 8 + [_i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_bwd": (_i, [_vp] * 13 + [_i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_decode_probe_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_fwd_probe": (_i, [_vp] * 7 + [_i, _i, _i, _i, _i, _vp]),
    "parallax_fwd_probe_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "parallax_step_host": (_i, [_vp] * 12 + [_i, _i, _i, _i, _i, _i, _vp]),
}


class PlxError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {parallax_strerror(code)} (code {code})")


class PlxLibraryMissing(ImportError):
    pass


def lib_path() -> str:
    return _LIB_PATH


def exported_symbols() -> list[str]:
    return list(_SIGNATURES)


def lib():
    """Load libparallax.so (once).  Raises PlxLibraryMissing if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise PlxLibraryMissing(
                f"{_LIB_PATH} is not built; run `python -m parallax_local_linear_fwd_b300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return PLX_FP32
    if t.dtype == torch.bfloat16:
        return PLX_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16")


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _check(code: int, where: str):
    if code != PLX_OK:
        raise PlxError(code, where)


def _shape(q):
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("q must be a [B, H, T, d] tensor")
    return tuple(int(x) for x in q.shape)


def _expect(name, t, shape, dtype, device, optional=False):
    """Checks one tensor argument against the shape, dtype and device the C
    ABI will assume for it; every pointer that reaches the library has passed
    this, so a mismatched tensor cannot make a kernel read or write past it."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected dtype {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _cuda_device(q):
    if q.device.type != "cuda":
        raise ValueError(f"tensors must be on a CUDA device, got {q.device}")
    return q.device


def _on(t):
    """The library launches on the current device: make it the tensors' own."""
    return torch.cuda.device(t.device)


def _expect_workspace(ws, nbytes, device):
    if ws is None:
        return
    if not isinstance(ws, torch.Tensor) or ws.device != device or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    if ws.numel() * ws.element_size() < nbytes:
        raise ValueError(f"workspace holds {ws.numel() * ws.element_size()} bytes, needs {nbytes}")


def _check_dtype(q):
    _dtype_code(q)
    return q.dtype


def _fwd_checks(q, k, v, P, out, lse, mu_k):
    B, H, T, d = _shape(q)
    dt = _check_dtype(q)
    dev = q.device
    for name, t in (("k", k), ("v", v)):
        _expect(name, t, (B, H, T, d), dt, dev)
    _expect("P", P, (H, d, d), torch.float32, dev)
    _expect("out", out, (B, H, T, d), dt, dev, optional=True)
    _expect("lse", lse, (B, H, T), torch.float32, dev, optional=True)
    _expect("mu_k", mu_k, (B, H, T, d), torch.float32, dev, optional=True)
    _cuda_device(q)
    return B, H, T, d


def parallax_fwd(q, k, v, P, out=None, lse=None, mu_k=None, stream=None):
    """Forward; returns (out, lse, mu_k).  q, k, v: [B,H,T,d] fp32/bf16 (CUDA)."""
    B, H, T, d = _fwd_checks(q, k, v, P, out, lse, mu_k)
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if mu_k is None:
        mu_k = torch.empty((B, H, T, d), dtype=torch.float32, device=q.device)
    with _on(q):
        _check(lib().parallax_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(lse), _ptr(mu_k),
                                  B, H, T, d, dt, _stream_ptr(stream)), "parallax_fwd")
    return out, lse, mu_k


def parallax_fwd_noalloc(q, k, v, P, out=None, lse=None, mu_k=None, stream=None):
    """Forward that allocates no device memory inside the library.

    For callers that cannot allocate (memory owned by another allocator, or a
    loop where an allocation would synchronise the device).  Pass preallocated
    out/lse/mu_k to keep this wrapper allocation-free too.  The library's
    fixed 32 MiB scratch limits the size; larger problems raise PlxError with
    PLX_ERR_TOO_LARGE.  Calls that overlap on the GPU race on that scratch.
    """
    B, H, T, d = _fwd_checks(q, k, v, P, out, lse, mu_k)
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device)
    if mu_k is None:
        mu_k = torch.empty((B, H, T, d), dtype=torch.float32, device=q.device)
    with _on(q):
        _check(lib().parallax_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(lse), _ptr(mu_k),
                                          B, H, T, d, dt, _stream_ptr(stream)), "parallax_fwd_noalloc")
    return out, lse, mu_k


def parallax_fwd_ws(q, k, v, P, out, lse, mu_k, workspace, stream=None):
    for name, t in (("out", out), ("lse", lse), ("mu_k", mu_k), ("workspace", workspace)):
        if t is None:
            raise ValueError(f"{name} is required")
    B, H, T, d = _fwd_checks(q, k, v, P, out, lse, mu_k)
    _expect_workspace(workspace, parallax_fwd_workspace_bytes(B, H, T, d, _dtype_code(q)), q.device)
    with _on(q):
        _check(lib().parallax_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(out), _ptr(lse), _ptr(mu_k),
                                     _ptr(workspace), B, H, T, d, _dtype_code(q), _stream_ptr(stream)),
               "parallax_fwd_ws")
    return out, lse, mu_k


def parallax_fwd_workspace_bytes(B, H, T, d, dtype) -> int:
    return int(lib().parallax_fwd_workspace_bytes(B, H, T, d, dtype))


def parallax_bwd_workspace_bytes(B, H, T, d, dtype) -> int:
    return int(lib().parallax_bwd_workspace_bytes(B, H, T, d, dtype))


def parallax_bwd(q, k, v, P, lse, mu_k, dout, dq=None, dk=None, dv=None, dP=None,
                 workspace=None, stream=None):
    """Backward of sum(dout * out); returns (dq, dk, dv, dP)."""
    B, H, T, d = _shape(q)
    dt = _dtype_code(q)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _expect(name, t, (B, H, T, d), q.dtype, dev)
    _expect("P", P, (H, d, d), torch.float32, dev)
    _expect("lse", lse, (B, H, T), torch.float32, dev)
    _expect("mu_k", mu_k, (B, H, T, d), torch.float32, dev)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(name, t, (B, H, T, d), q.dtype, dev, optional=True)
    _expect("dP", dP, (H, d, d), torch.float32, dev, optional=True)
    _cuda_device(q)
    if workspace is not None:
        _expect_workspace(workspace, parallax_bwd_workspace_bytes(B, H, T, d, dt), dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dP = torch.empty_like(P) if dP is None else dP
    with _on(q):
        _check(lib().parallax_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(lse), _ptr(mu_k),
                                  _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dP), _ptr(workspace),
                                  B, H, T, d, dt, _stream_ptr(stream)), "parallax_bwd")
    return dq, dk, dv, dP


def parallax_fwd_bwd_workspace_bytes(B, H, T, d, dtype) -> int:
    return int(lib().parallax_fwd_bwd_workspace_bytes(B, H, T, d, dtype))


def parallax_fwd_bwd(q, k, v, P, dout, out=None, lse=None, mu_k=None, dq=None, dk=None, dv=None, dP=None,
                     workspace=None, stream=None):
    """Forward and backward of one step in one call (one workspace: the
    backward reuses the forward's f16 operand copies).  Returns
    (out, lse, mu_k, dq, dk, dv, dP), equal to parallax_fwd then parallax_bwd."""
    B, H, T, d = _shape(q)
    dt = _dtype_code(q)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("dout", dout)):
        _expect(name, t, (B, H, T, d), q.dtype, dev)
    _expect("P", P, (H, d, d), torch.float32, dev)
    for name, t in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(name, t, (B, H, T, d), q.dtype, dev, optional=True)
    _expect("lse", lse, (B, H, T), torch.float32, dev, optional=True)
    _expect("mu_k", mu_k, (B, H, T, d), torch.float32, dev, optional=True)
    _expect("dP", dP, (H, d, d), torch.float32, dev, optional=True)
    _cuda_device(q)
    if workspace is not None:
        _expect_workspace(workspace, parallax_fwd_bwd_workspace_bytes(B, H, T, d, dt), dev)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, T), dtype=torch.float32, device=dev) if lse is None else lse
    mu_k = torch.empty((B, H, T, d), dtype=torch.float32, device=dev) if mu_k is None else mu_k
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dP = torch.empty_like(P) if dP is None else dP
    with _on(q):
        _check(lib().parallax_fwd_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(dout), _ptr(out), _ptr(lse),
                                      _ptr(mu_k), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dP), _ptr(workspace),
                                      B, H, T, d, dt, _stream_ptr(stream)), "parallax_fwd_bwd")
    return out, lse, mu_k, dq, dk, dv, dP


def parallax_fwd_probe_workspace_bytes(B, H, T, d, dtype) -> int:
    return int(lib().parallax_fwd_probe_workspace_bytes(B, H, T, d, dtype))


def parallax_fwd_probe(q, k, v, rho, out=None, lse=None, workspace=None, stream=None):
    """One-pass forward with a given probe rho [B,H,T,d] (bf16): o = o^SA - Sigma_KV rho.
    Returns (out, lse)."""
    B, H, T, d = _shape(q)
    dt = _check_dtype(q)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("rho", rho)):
        _expect(name, t, (B, H, T, d), dt, dev)
    _expect("out", out, (B, H, T, d), dt, dev, optional=True)
    _expect("lse", lse, (B, H, T), torch.float32, dev, optional=True)
    _cuda_device(q)
    if workspace is not None:
        _expect_workspace(workspace, parallax_fwd_probe_workspace_bytes(B, H, T, d, _dtype_code(q)), dev)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    with _on(q):
        _check(lib().parallax_fwd_probe(_ptr(q), _ptr(k), _ptr(v), _ptr(rho), _ptr(out), _ptr(lse), _ptr(workspace),
                                        B, H, T, d, _dtype_code(q), _stream_ptr(stream)), "parallax_fwd_probe")
    return out, lse


def parallax_decode_workspace_bytes(B, H, Lmax, d, dtype) -> int:
    return int(lib().parallax_decode_workspace_bytes(B, H, Lmax, d, dtype))


def parallax_decode(q, k_cache, v_cache, P, lens=None, out=None, lse=None, workspace=None, stream=None):
    """Decode step: q [B,H,d] against caches [B,H,Lmax,d] (fp32/bf16, CUDA);
    lens: int32 [B] valid keys per sequence (None: Lmax).  Returns (out, lse)."""
    if not isinstance(k_cache, torch.Tensor) or k_cache.dim() != 4:
        raise ValueError("the caches must be [B, H, Lmax, d] tensors")
    B, H, Lmax, d = (int(x) for x in k_cache.shape)
    dt = _dtype_code(k_cache)
    dev = k_cache.device
    _expect("q", q, (B, H, d), k_cache.dtype, dev)
    _expect("v_cache", v_cache, (B, H, Lmax, d), k_cache.dtype, dev)
    _expect("k_cache", k_cache, (B, H, Lmax, d), k_cache.dtype, dev)
    _expect("P", P, (H, d, d), torch.float32, dev)
    _expect("lens", lens, (B,), torch.int32, dev, optional=True)
    _expect("out", out, (B, H, d), k_cache.dtype, dev, optional=True)
    _expect("lse", lse, (B, H), torch.float32, dev, optional=True)
    _cuda_device(k_cache)
    if workspace is not None:
        _expect_workspace(workspace, parallax_decode_workspace_bytes(B, H, Lmax, d, dt), dev)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    with _on(k_cache):
        _check(lib().parallax_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), _ptr(P), _ptr(out),
                                     _ptr(lse), _ptr(workspace), B, H, Lmax, d, dt, _stream_ptr(stream)),
               "parallax_decode")
    return out, lse


def parallax_decode_probe_workspace_bytes(B, H, Lmax, d, dtype) -> int:
    return int(lib().parallax_decode_probe_workspace_bytes(B, H, Lmax, d, dtype))


def parallax_decode_probe(q, k_cache, v_cache, rho, lens=None, out=None, lse=None, workspace=None, stream=None):
    """Decode step with a given probe rho [B,H,d]: q [B,H,d] against caches
    [B,H,Lmax,d] (bf16, CUDA), o = o^SA - Sigma_KV rho in one pass over the
    keys and values; lens: int32 [B] (None: Lmax).  Returns (out, lse)."""
    if not isinstance(k_cache, torch.Tensor) or k_cache.dim() != 4:
        raise ValueError("the caches must be [B, H, Lmax, d] tensors")
    B, H, Lmax, d = (int(x) for x in k_cache.shape)
    dt = _dtype_code(k_cache)
    dev = k_cache.device
    _expect("q", q, (B, H, d), k_cache.dtype, dev)
    _expect("rho", rho, (B, H, d), k_cache.dtype, dev)
    _expect("v_cache", v_cache, (B, H, Lmax, d), k_cache.dtype, dev)
    _expect("lens", lens, (B,), torch.int32, dev, optional=True)
    _expect("out", out, (B, H, d), k_cache.dtype, dev, optional=True)
    _expect("lse", lse, (B, H), torch.float32, dev, optional=True)
    _cuda_device(k_cache)
    if workspace is not None:
        _expect_workspace(workspace, parallax_decode_probe_workspace_bytes(B, H, Lmax, d, dt), dev)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    with _on(k_cache):
        _check(lib().parallax_decode_probe(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), _ptr(rho), _ptr(out),
                                           _ptr(lse), _ptr(workspace), B, H, Lmax, d, dt, _stream_ptr(stream)),
               "parallax_decode_probe")
    return out, lse


def parallax_step_host(q, k, v, P, dout, out=None, dq=None, dk=None, dv=None, dP=None, lse=None, mu_k=None,
                       chunks=0, stream=None):
    """Forward + backward from host (CPU) tensors, copies overlapped with compute.

    q, k, v, dout: [B,H,T,d] float32/bfloat16 CPU tensors (pinned for overlap); P [H,d,d] float32.
    Outputs (allocated pinned when None): out, dq, dk, dv like q, dP like P.  lse [B,H,T] and
    mu_k [B,H,T,d] float32 are returned only when passed in.  The call is asynchronous on
    `stream`: synchronize it before reading the outputs.  Returns (out, dq, dk, dv, dP, lse, mu_k).
    """
    B, H, T, d = _shape(q)
    dt = _check_dtype(q)
    cpu = torch.device("cpu")
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout)):
        _expect(name, t, (B, H, T, d), dt, cpu)
    _expect("P", P, (H, d, d), torch.float32, cpu)
    for name, t in (("out", out), ("dq", dq), ("dk", dk), ("dv", dv)):
        _expect(name, t, (B, H, T, d), dt, cpu, optional=True)
    _expect("dP", dP, (H, d, d), torch.float32, cpu, optional=True)
    _expect("lse", lse, (B, H, T), torch.float32, cpu, optional=True)
    _expect("mu_k", mu_k, (B, H, T, d), torch.float32, cpu, optional=True)

    def alloc(like):
        return torch.empty(like.shape, dtype=like.dtype).pin_memory()

    out = alloc(q) if out is None else out
    dq = alloc(q) if dq is None else dq
    dk = alloc(k) if dk is None else dk
    dv = alloc(v) if dv is None else dv
    dP = alloc(P) if dP is None else dP
    _check(lib().parallax_step_host(_ptr(q), _ptr(k), _ptr(v), _ptr(P), _ptr(dout), _ptr(out), _ptr(lse),
                                    _ptr(mu_k), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dP), int(chunks),
                                    B, H, T, d, _dtype_code(q), _stream_ptr(stream)), "parallax_step_host")
    return out, dq, dk, dv, dP, lse, mu_k


def parallax_last_device_error(stream=None):
    """Synchronize `stream` and return (code, detail) of the device watchdog."""
    detail = ctypes.c_uint(0)
    code = lib().parallax_last_device_error(_stream_ptr(stream), ctypes.byref(detail))
    return int(code), int(detail.value)


def parallax_set_path(path: int) -> int:
    return int(lib().parallax_set_path(path))


def parallax_set_persistent_ctas(ctas: int) -> int:
    """Cap on the CTAs of the persistent kernels (0: the default); returns the
    previous cap.  A test hook: a small cap makes each CTA run many items."""
    prev = int(lib().parallax_set_persistent_ctas(int(ctas)))
    if prev < 0:
        raise ValueError(f"parallax_set_persistent_ctas: ctas must be >= 0, got {ctas}")
    return prev


def parallax_set_wait_limit(cycles: int) -> None:
    """Bounded-wait limit of the tensor-core kernels on the current device,
    in SM cycles (<= 0: the default, about two seconds).  A test hook for the
    watchdog path: a short limit makes waits time out on purpose."""
    _check(lib().parallax_set_wait_limit(int(cycles)), "parallax_set_wait_limit")


def parallax_strerror(code: int) -> str:
    try:
        return lib().parallax_strerror(code).decode()
    except PlxLibraryMissing:
        return f"status {code}"


def parallax_launch_count() -> int:
    """Total kernel launches the library has made in this process."""
    return int(lib().parallax_launch_count())


def parallax_timing_enable(on: bool) -> bool:
    return bool(lib().parallax_timing_enable(1 if on else 0))


def parallax_timing_collect() -> int:
    n = int(lib().parallax_timing_collect())
    if n < 0:
        raise PlxError(-n, "parallax_timing_collect")
    return n


def parallax_timing_get(i: int):
    name = ctypes.c_char_p()
    ms = ctypes.c_double()
    cnt = ctypes.c_longlong()
    _check(lib().parallax_timing_get(i, ctypes.byref(name), ctypes.byref(ms), ctypes.byref(cnt)),
           "parallax_timing_get")
    return name.value.decode(), float(ms.value), int(cnt.value)


def parallax_timing_reset() -> None:
    lib().parallax_timing_reset()


def kernel_times() -> dict:
    """{kernel name: (total ms, launches)} of the timed launches so far."""
    n = parallax_timing_collect()
    out = {}
    for i in range(n):
        name, ms, cnt = parallax_timing_get(i)
        if cnt:
            out[name] = (ms, cnt)
    return out
