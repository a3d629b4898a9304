"""Exact attention for GB300 (sm_103a): thin Python binding of libfa.so.

Every function here only marshals torch tensors into the C ABI declared in
``include/fa.h`` (device pointers, sizes, the current CUDA stream) and checks
the returned status; all arithmetic runs in the library's CUDA kernels.  There
is no fallback: if ``libfa.so`` is missing or a call fails, an exception is
raised.

Functions keep the C names (see ``__all__``).  Every tensor a call touches,
inputs, caller-supplied outputs and workspaces alike, is checked for device,
dtype, shape and contiguity before the library is called, since the kernels
trust the sizes they are given.  A call runs on the device of its ``q`` and
on that device's current stream unless ``stream`` is given.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "FaError", "library_path", "load_library", "fa_fwd", "fa_fwd_varlen", "fa_fwd_paged",
    "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "fa_fwd_fp8", "fa_fwd_varlen_fp8",
    "fa_bwd", "fa_bwd_varlen", "fa_bwd_workspace_size",
    "fa_decode_paged", "fa_decode_paged_noalloc", "fa_decode_workspace_size",
    "fa_status_string", "fa_device_status", "fa_last_device_status", "new_workspace",
    "FA_WORKSPACE_HEADER_BYTES",
    "fa_version", "FA_DEV_TIMEOUT", "FA_DEV_BAD_BLOCK", "FA_DEV_BAD_CTX", "FA_DEV_BAD_SEQLEN",
    "FA_DEV_BAD_INDEX", "FA_DEV_SMEM_ALIGN",
]

FA_OK = 0
FA_DEV_TIMEOUT = 1
FA_DEV_BAD_BLOCK = 2
FA_DEV_BAD_CTX = 4
FA_DEV_BAD_SEQLEN = 8
FA_DEV_BAD_INDEX = 16   # checked build only
FA_DEV_SMEM_ALIGN = 32  # a kernel found its shared memory not 1 KiB aligned
FA_WORKSPACE_HEADER_BYTES = 256   # control block at the start of a decode / split-KV workspace

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {status} ({fa_status_string(status)})")


def library_path() -> str:
    """libfa.so, or the checked build libfa_checked.so when FA_CHECKED=1."""
    name = "libfa_checked.so" if os.environ.get("FA_CHECKED") == "1" else "libfa.so"
    return os.path.join(_PKG, name)


def load_library() -> ctypes.CDLL:
    """Load libfa.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m exact_attention_33_gb300.build` "
                "(add --checked for the checked build, or call __graft_entry__.build()); "
                "there is no non-CUDA fallback")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        lib.fa_fwd.restype = i
        lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        lib.fa_fwd_varlen.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, i, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_fwd_varlen_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, f, f, i, vp]
        lib.fa_fwd_varlen_fp8.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
        lib.fa_bwd.restype = i
        lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                      i, vp, sz, vp]
        lib.fa_bwd_varlen.restype = i
        lib.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i]
        lib.fa_fwd_splitkv_workspace_size.restype = sz
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]
        lib.fa_fwd_splitkv.restype = i
        lib.fa_fwd_paged.argtypes = [vp, vp, vp, vp, i, vp, vp, i, i, i, i, i, i, i, i, i, f, i,
                                     vp, vp, vp]
        lib.fa_fwd_paged.restype = i
        lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.fa_decode_workspace_size.restype = sz
        lib.fa_decode_paged.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f, vp, vp,
                                        vp, sz, vp]
        lib.fa_decode_paged.restype = i
        lib.fa_decode_paged_noalloc.argtypes = [vp, vp, vp, vp, i, vp, i, i, i, i, i, i, i, f,
                                                vp, vp, vp]
        lib.fa_decode_paged_noalloc.restype = i
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), i]
        lib.fa_device_status.restype = i
        lib.fa_last_device_status.argtypes = [vp]
        lib.fa_last_device_status.restype = i
        lib.fa_selftest_wait_timeout.argtypes = [vp, vp]
        lib.fa_selftest_wait_timeout.restype = i
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i
        _lib = lib
        return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def fa_version() -> int:
    return int(load_library().fa_version())


def fa_selftest_wait_timeout(stream=None) -> int:
    """Run the bounded-wait self-test; returns the wait's result (0 = it gave
    up, as intended).  FA_DEV_TIMEOUT is set in the status word afterwards."""
    torch = _torch()
    res = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rc = load_library().fa_selftest_wait_timeout(_ptr(res), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError("fa_selftest_wait_timeout", rc)
    torch.cuda.synchronize()
    return int(res.item())


def fa_device_status(clear: bool = True) -> int:
    """Sticky device status word (FA_DEV_* bits); synchronises the device."""
    v = ctypes.c_uint(0)
    rc = load_library().fa_device_status(ctypes.byref(v), 1 if clear else 0)
    if rc != FA_OK:
        raise FaError("fa_device_status", rc)
    return int(v.value)


def fa_last_device_status(workspace) -> int:
    """FA_DEV_* bits of the last call that finished on ``workspace`` (a
    decode or split-KV workspace).  Read it after that call has completed
    (synchronise its stream first); it does not wait for other streams."""
    torch = _torch()
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda \
            or workspace.numel() * workspace.element_size() < FA_WORKSPACE_HEADER_BYTES:
        raise ValueError("workspace must be a CUDA tensor of at least "
                         f"{FA_WORKSPACE_HEADER_BYTES} bytes")
    with torch.cuda.device(workspace.device):
        rc = load_library().fa_last_device_status(_ptr(workspace))
    if rc < 0:
        raise FaError("fa_last_device_status", rc)
    return int(rc)


def new_workspace(nbytes: int, device=None):
    """A decode or split-KV workspace of ``nbytes`` bytes, zero-filled as the
    library requires before its first call."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), FA_WORKSPACE_HEADER_BYTES), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


# ----------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _stream_handle(stream=None, device=None):
    torch = _torch()
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(int(s.cuda_stream))


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else int(t.data_ptr()))


def _check_bf16_cuda(name, t, ndim, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def _check_tensor(name, t, shape, dtype, device):
    """A tensor the kernels read or write with exactly this shape and dtype."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}")
    if tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor of shape {tuple(shape)}")


def _check_int32(name, t, device, ndim=1, numel=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != torch.int32 or t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D int32 tensor")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} values")


def _workspace(t, need, device, minimum=1, zero=False):
    """The caller's workspace (a 1-D uint8 tensor, its length in bytes), or a
    new one of at least ``need`` bytes (zero-filled with ``zero``: decode and
    split-KV workspaces start with a control block that must be zero)."""
    torch = _torch()
    if t is None:
        alloc = torch.zeros if zero else torch.empty
        return alloc(max(need, minimum), dtype=torch.uint8, device=device)
    if not isinstance(t, torch.Tensor) or t.device != device or t.dtype != torch.uint8 \
            or t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"workspace must be a contiguous 1-D uint8 tensor on {device}")
    return t


def _outputs(q_like_shape, lse_shape, out, lse, want_lse, device):
    torch = _torch()
    if out is None:
        out = torch.empty(q_like_shape, dtype=torch.bfloat16, device=device)
    else:
        _check_tensor("out", out, q_like_shape, torch.bfloat16, device)
    if lse is None and want_lse:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=device)
    elif lse is not None:
        _check_tensor("lse", lse, lse_shape, torch.float32, device)
    return out, lse


def _scale(scale, d):
    return float(1.0 / math.sqrt(d)) if scale is None else float(scale)


# ----------------------------------------------------------------- calls

def fa_fwd(q, k, v, causal=False, scale=None, out=None, lse=None, want_lse=True, stream=None):
    """Dense prefill.  q [B,N,H,d], k/v [B,N,Hkv,d] bf16 CUDA tensors.

    Returns (out [B,N,H,d] bf16, lse [B,H,N] fp32 or None).
    """
    torch = _torch()
    _check_bf16_cuda("q", q, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v)):
        _check_bf16_cuda(name, t, 4, dev)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d] matching q")
    out, lse = _outputs(q.shape, (B, H, N), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv,
                                   N, d, _scale(scale, d), 1 if causal else 0,
                                   _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd", rc)
    return out, lse


def fa_bwd_workspace_size(B, H, N) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N))


def fa_bwd(q, k, v, out, lse, dout, causal=False, scale=None, dq=None, dk=None, dv=None,
           workspace=None, stream=None):
    """Gradient of dense attention.  q, out, dout [B,N,H,d]; k, v [B,N,Hkv,d]
    bf16 CUDA tensors; lse [B,H,N] fp32 from fa_fwd.  Returns (dq, dk, dv)."""
    torch = _torch()
    _check_bf16_cuda("q", q, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_bf16_cuda(name, t, 4, dev)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or out.shape != q.shape \
            or dout.shape != q.shape:
        raise ValueError("shapes must be q/out/dout [B,N,H,d], k/v [B,N,Hkv,d]")
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    grads = []
    for name, g, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if g is None:
            g = torch.empty_like(like)
        else:
            _check_tensor(name, g, like.shape, torch.bfloat16, dev)
        grads.append(g)
    dq, dk, dv = grads
    workspace = _workspace(workspace, fa_bwd_workspace_size(B, H, N), dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                   _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d,
                                   _scale(scale, d), 1 if causal else 0, _ptr(workspace),
                                   workspace.numel(), _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_bwd", rc)
    return dq, dk, dv


def fa_bwd_varlen(q, k, v, out, lse, dout, cu_seqlens, max_seqlen, causal=False, scale=None,
                  dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradient of a packed varlen batch.  q, out, dout [T,H,d]; k, v [T,Hkv,d]
    bf16 CUDA tensors; lse [H,T] fp32 from fa_fwd_varlen; cu_seqlens int32
    [S+1] on the device.  Returns (dq, dk, dv); rows outside every sequence
    are left as they were."""
    torch = _torch()
    _check_bf16_cuda("q", q, 3)
    dev = q.device
    for name, t in (("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_bf16_cuda(name, t, 3, dev)
    _check_int32("cu_seqlens", cu_seqlens, dev)
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must hold num_seqs + 1 offsets")
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape or out.shape != q.shape \
            or dout.shape != q.shape:
        raise ValueError("shapes must be q/out/dout [T,H,d], k/v [T,Hkv,d]")
    _check_tensor("lse", lse, (H, T), torch.float32, dev)
    grads = []
    for name, g, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if g is None:
            g = torch.empty_like(like)
        else:
            _check_tensor(name, g, like.shape, torch.bfloat16, dev)
        grads.append(g)
    dq, dk, dv = grads
    S = cu_seqlens.numel() - 1
    workspace = _workspace(workspace, fa_bwd_workspace_size(S, H, min(int(max_seqlen), T)), dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_bwd_varlen(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
            _ptr(dv), _ptr(cu_seqlens), S, T, int(max_seqlen), H, Hkv, d, _scale(scale, d),
            1 if causal else 0, _ptr(workspace), workspace.numel(), _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_bwd_varlen", rc)
    return dq, dk, dv


def fa_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, causal=False, scale=None, out=None,
               lse=None, want_lse=True, stream=None):
    """Dense prefill on e4m3 codes.  q [B,N,H,d], k/v [B,N,Hkv,d] uint8 CUDA
    tensors holding e4m3 bits; per-tensor descales.  Returns (out bf16, lse)."""
    torch = _torch()
    dev = q.device if isinstance(q, torch.Tensor) else None
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != dev \
                or t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != 4 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D uint8/e4m3 CUDA tensor on the "
                             "device of q")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d] matching q")
    out, lse = _outputs((B, N, H, d), (B, H, N), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H,
                                       Hkv, N, d, _scale(scale, d), float(q_descale),
                                       float(k_descale), float(v_descale), 1 if causal else 0,
                                       _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd_fp8", rc)
    return out, lse


def _check_fp8(name, t, ndim, dev):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != dev \
            or t.dtype not in (torch.uint8, torch.float8_e4m3fn) or t.dim() != ndim \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D uint8/e4m3 CUDA tensor on the "
                         "device of q")


def fa_fwd_varlen_fp8(q, k, v, cu_seqlens, max_seqlen, q_descale, k_descale, v_descale,
                      causal=False, scale=None, out=None, lse=None, want_lse=True, stream=None):
    """Packed varlen prefill on e4m3 codes.  q [T,H,d], k/v [T,Hkv,d] uint8
    CUDA tensors holding e4m3 bits, cu_seqlens int32 [S+1] on the device;
    per-tensor descales.  Returns (out [T,H,d] bf16, lse [H,T] fp32 or None)."""
    torch = _torch()
    dev = q.device if isinstance(q, torch.Tensor) else None
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_fp8(name, t, 3, dev)
    _check_int32("cu_seqlens", cu_seqlens, dev)
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must hold num_seqs + 1 offsets")
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, d] matching q")
    out, lse = _outputs((T, H, d), (H, T), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd_varlen_fp8(
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens),
            cu_seqlens.numel() - 1, T, int(max_seqlen), H, Hkv, d, _scale(scale, d),
            float(q_descale), float(k_descale), float(v_descale), 1 if causal else 0,
            _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd_varlen_fp8", rc)
    return out, lse


def fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits=0) -> int:
    return int(load_library().fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits))


def fa_fwd_splitkv(q, k, v, causal=False, scale=None, num_splits=0, out=None, lse=None,
                   workspace=None, want_lse=True, stream=None):
    """Dense prefill with split-KV partial states and a combine (for small
    B * H).  Same layouts as :func:`fa_fwd`."""
    torch = _torch()
    _check_bf16_cuda("q", q, 4)
    dev = q.device
    for name, t in (("k", k), ("v", v)):
        _check_bf16_cuda(name, t, 4, dev)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d] matching q")
    workspace = _workspace(workspace, fa_fwd_splitkv_workspace_size(B, H, N, d, num_splits),
                           dev, 256, zero=True)
    out, lse = _outputs(q.shape, (B, H, N), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B,
                                           H, Hkv, N, d, _scale(scale, d), 1 if causal else 0,
                                           int(num_splits), _ptr(workspace), workspace.numel(),
                                           _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd_splitkv", rc)
    return out, lse


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, causal=False, scale=None, out=None,
                  lse=None, want_lse=True, stream=None):
    """Packed varlen prefill.  q [T,H,d], k/v [T,Hkv,d], cu_seqlens int32 [S+1] on device.

    Returns (out [T,H,d] bf16, lse [H,T] fp32 or None).
    """
    torch = _torch()
    _check_bf16_cuda("q", q, 3)
    dev = q.device
    for name, t in (("k", k), ("v", v)):
        _check_bf16_cuda(name, t, 3, dev)
    _check_int32("cu_seqlens", cu_seqlens, dev)
    if cu_seqlens.numel() < 1:
        raise ValueError("cu_seqlens must hold num_seqs + 1 offsets")
    T, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (T, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [T, Hkv, d] matching q")
    out, lse = _outputs(q.shape, (H, T), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                          _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                          int(max_seqlen), H, Hkv, d, _scale(scale, d),
                                          1 if causal else 0, _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd_varlen", rc)
    return out, lse


def _check_pools(k_pool, v_pool, dev):
    _check_bf16_cuda("k_pool", k_pool, 4, dev)
    _check_bf16_cuda("v_pool", v_pool, 4, dev)
    if v_pool.shape != k_pool.shape:
        raise ValueError("k_pool and v_pool must have the same shape [num_blocks,16,Hkv,d]")
    return k_pool.shape


def fa_fwd_paged(q, k_pool, v_pool, block_table, ctx_lens, cu_seqlens_q, max_seqlen_q,
                 max_ctx_len, causal=True, scale=None, out=None, lse=None, want_lse=True,
                 stream=None):
    """Query chunks [Tq,H,d] against a paged KV cache (chunked prefill).

    pools [num_blocks,16,Hkv,d] bf16; block_table int32 [batch,max_blocks];
    ctx_lens int32 [batch]; cu_seqlens_q int32 [batch+1]; all on the device.
    Returns (out [Tq,H,d] bf16, lse [H,Tq] fp32 or None).
    """
    torch = _torch()
    _check_bf16_cuda("q", q, 3)
    dev = q.device
    num_blocks, block_size, Hkv, dp = _check_pools(k_pool, v_pool, dev)
    _check_int32("block_table", block_table, dev, ndim=2)
    batch = block_table.shape[0]
    _check_int32("ctx_lens", ctx_lens, dev, numel=batch)
    _check_int32("cu_seqlens_q", cu_seqlens_q, dev, numel=batch + 1)
    Tq, H, d = q.shape
    if dp != d:
        raise ValueError("the pools' head size must match q")
    out, lse = _outputs(q.shape, (H, Tq), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_fwd_paged(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), block_table.shape[1],
            _ptr(ctx_lens), _ptr(cu_seqlens_q), batch, Tq, int(max_seqlen_q),
            int(max_ctx_len), H, Hkv, d, block_size, num_blocks, _scale(scale, d),
            1 if causal else 0, _ptr(out), _ptr(lse), _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_fwd_paged", rc)
    return out, lse


def fa_decode_workspace_size(batch, H, Hkv, d, max_ctx_len, block_size=16) -> int:
    return int(load_library().fa_decode_workspace_size(batch, H, Hkv, d, max_ctx_len,
                                                       block_size))


def _decode_args(q, k_pool, v_pool, block_table, ctx_lens):
    _check_bf16_cuda("q", q, 3)
    dev = q.device
    num_blocks, block_size, Hkv, dp = _check_pools(k_pool, v_pool, dev)
    batch, H, d = q.shape
    if dp != d:
        raise ValueError("the pools' head size must match q")
    _check_int32("block_table", block_table, dev, ndim=2)
    if block_table.shape[0] != batch:
        raise ValueError("block_table must have one row per sequence of q")
    _check_int32("ctx_lens", ctx_lens, dev, numel=batch)
    return dev, batch, H, Hkv, d, num_blocks, block_size


def fa_decode_paged(q, k_pool, v_pool, block_table, ctx_lens, max_ctx_len, scale=None,
                    out=None, lse=None, workspace=None, want_lse=True, stream=None):
    """Paged GQA flash-decoding.

    q [batch,H,d]; pools [num_blocks,block_size,Hkv,d] bf16; block_table int32
    [batch, max_blocks]; ctx_lens int32 [batch]; all on the device.
    Returns (out [batch,H,d] bf16, lse [batch,H] fp32 or None).
    """
    torch = _torch()
    dev, batch, H, Hkv, d, num_blocks, block_size = _decode_args(q, k_pool, v_pool,
                                                                 block_table, ctx_lens)
    workspace = _workspace(
        workspace, fa_decode_workspace_size(batch, H, Hkv, d, max_ctx_len, block_size), dev, 256,
        zero=True)
    out, lse = _outputs(q.shape, (batch, H), out, lse, want_lse, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_decode_paged(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), block_table.shape[1],
            _ptr(ctx_lens), int(max_ctx_len), batch, H, Hkv, d, block_size, num_blocks,
            _scale(scale, d), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_decode_paged", rc)
    return out, lse


FA_DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20


def fa_decode_paged_noalloc(q, k_pool, v_pool, block_table, ctx_lens, max_ctx_len, *, out,
                            lse=None, scale=None, stream=None):
    """Paged decode that allocates nothing on the device, for callers that
    cannot call cudaMalloc (a plugin whose host framework owns all device
    memory, or a decode loop that must avoid the implicit synchronisation of
    cudaMalloc/cudaFree).  The split partial states live in the library's
    static scratch array of FA_DECODE_NOALLOC_SCRATCH_BYTES; larger requests
    are rejected.  The caller passes ``out`` (and optionally ``lse``); calls
    whose kernels overlap on the GPU race on the shared scratch."""
    torch = _torch()
    dev, batch, H, Hkv, d, num_blocks, block_size = _decode_args(q, k_pool, v_pool,
                                                                 block_table, ctx_lens)
    _check_tensor("out", out, q.shape, torch.bfloat16, dev)
    if lse is not None:
        _check_tensor("lse", lse, (batch, H), torch.float32, dev)
    with torch.cuda.device(dev):
        rc = load_library().fa_decode_paged_noalloc(
            _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(block_table), block_table.shape[1],
            _ptr(ctx_lens), int(max_ctx_len), batch, H, Hkv, d, block_size, num_blocks,
            _scale(scale, d), _ptr(out), _ptr(lse), _stream_handle(stream, dev))
    if rc != FA_OK:
        raise FaError("fa_decode_paged_noalloc", rc)
    return out, lse
