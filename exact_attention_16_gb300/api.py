"""Python binding of the C ABI in include/fa.h (ctypes; marshalling only).

Every function here has the name of the C entry point it wraps. Tensors are
PyTorch CUDA tensors; the binding checks dtype, device, shape and contiguity,
passes raw device pointers and the current CUDA stream, and raises
:class:`FAError` on a non-zero status. There is no fallback: if the compiled
library is missing, loading it raises.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "FAError",
    "lib",
    "library_path",
    "fa_fwd",
    "fa_fwd_strided",
    "fa_merge",
    "fa_fwd_decode",
    "fa_decode_workspace_size",
    "fa_fwd_decode_noalloc",
    "fa_fwd_host",
    "fa_fwd_host_workspace_size",
    "fa_fwd_host_plan",
    "fa_decode_splits",
    "fa_status",
    "fa_status_string",
    "fa_version",
    "fa_debug_set_fault",
    "fa_debug_set_schedule",
    "fa_fwd_schedule",
    "fa_fwd_work_items",
    "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_lib", "libfa_gb300.so")
_lock = threading.Lock()
_lib = None

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_DTYPE_FP16, FA_DTYPE_BF16 = 0, 1

# name -> (restype, argtypes); the entry points include/fa.h declares
EXPORTED_SYMBOLS = {
    "fa_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                              ctypes.c_void_p]),
    "fa_fwd_strided": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int,
                                      # four `const long long[3]` stride arrays, passed by address
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                      ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_merge": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    "fa_fwd_decode": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]),
    "fa_decode_workspace_size": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_fwd_decode_noalloc": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_void_p]),
    "fa_status": (ctypes.c_int, [ctypes.c_void_p]),
    "fa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "fa_version": (ctypes.c_int, []),
    "fa_debug_set_fault": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "fa_debug_set_schedule": (ctypes.c_int, [ctypes.c_int]),
    "fa_fwd_host_workspace_size": (ctypes.c_int, [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_ulonglong)]),
    "fa_decode_splits": (ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.POINTER(ctypes.c_int)]),
    "fa_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 6
                    + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_ulonglong,
                       ctypes.c_void_p]),
    "fa_fwd_schedule": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.POINTER(ctypes.c_int)]),
    "fa_fwd_work_items": (ctypes.c_int, [ctypes.c_int] * 8 + [ctypes.c_void_p, ctypes.c_int,
                                                              ctypes.POINTER(ctypes.c_int),
                                                              ctypes.POINTER(ctypes.c_int)]),
    "fa_fwd_host_plan": (ctypes.c_int, [ctypes.c_int] * 7 + [ctypes.c_void_p, ctypes.c_int,
                                                             ctypes.POINTER(ctypes.c_int)]),
}


class FAError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        name = lib().fa_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{what}: {name}" if what else name)


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(_LIB_PATH):
                    raise ImportError(
                        f"{_LIB_PATH} is missing: build it with `python -m exact_attention_16_gb300.build`")
                handle = ctypes.CDLL(_LIB_PATH)
                for name, (res, args) in EXPORTED_SYMBOLS.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def _stream_handle(stream, device_index=None):
    """cudaStream_t of ``stream``, or of the current stream of the device."""
    import torch

    if stream is None:
        if device_index is None:
            device_index = torch.cuda.current_device()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)   # cheap path, no Stream object
        if raw is not None:
            return ctypes.c_void_p(raw(device_index))
        stream = torch.cuda.current_stream(device_index)
    return ctypes.c_void_p(stream.cuda_stream)


def _call_on(device_index, fn):
    """Runs ``fn`` with CUDA device ``device_index`` current (switching only
    when another device is)."""
    import torch

    if torch.cuda.current_device() == device_index:
        return fn()
    with torch.cuda.device(device_index):
        return fn()


_LL12 = ctypes.c_longlong * 12


def _dtype_code(t):
    import torch

    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float16:
        return FA_DTYPE_FP16
    raise TypeError(f"unsupported dtype {t.dtype}; expected torch.bfloat16 or torch.float16")


def _check_result(name, t, shape, dtype, device):
    """A caller-supplied result buffer: a contiguous CUDA tensor of exactly
    ``shape`` and ``dtype`` on ``device`` (the kernels write every element of
    that shape, so anything smaller would be overrun)."""
    import torch

    if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != device or tuple(t.shape) != tuple(shape)
            or t.dtype != dtype or not t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor of shape {tuple(shape)} on {device}")


def _check_workspace(ws, device):
    import torch

    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous CUDA tensor on {device}")


def _check_qkv_device(q, k, v):
    """q, k, v: contiguous 4-D CUDA tensors of one dtype on one device, k and
    v of one shape (B, Sk, Hkv, D) matching q's batch and head dimension."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
    if not (q.dtype == k.dtype == v.dtype) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must share one dtype and device")
    if tuple(v.shape) != tuple(k.shape) or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3]:
        raise ValueError("k and v must be (B, Sk, Hkv, D) matching q")


def fa_fwd(q, k, v, *, scale=None, causal=False, out=None, lse=None, return_lse=True, stream=None):
    """Attention forward: returns (O, LSE) (LSE is None if return_lse is False
    and no ``lse`` buffer is given).

    q: (B, Sq, Hq, D); k, v: (B, Sk, Hkv, D) CUDA tensors of one 16-bit dtype
    on one device, indexed (batch, seq, head, d). Any strides are accepted as
    long as d is contiguous and the other strides are multiples of 8
    elements (so ``x.transpose(1, 2)`` of a (B, H, S, D) tensor works as is).
    ``scale`` defaults to 1/sqrt(D). ``causal`` selects the bottom-right
    aligned mask (query i sees key j iff j <= i + Sk - Sq). ``out`` (any
    such strides) and ``lse`` (contiguous (B, Hq, Sq) float32) may be given.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be 4-D (batch, seq, heads, head_dim)")
        if t.stride(3) != 1:
            raise ValueError(f"{name}: the head dimension must be contiguous")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k and v must be on one device")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be (B, Sk, Hkv, D) matching q")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=q.dtype, device=q.device)
    elif tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype or out.device != q.device or out.stride(3) != 1:
        raise ValueError("out must be a (B, Sq, Hq, D) tensor like q with a contiguous head dimension")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    elif lse is not None and (tuple(lse.shape) != (B, Hq, Sq) or lse.dtype != torch.float32
                              or lse.device != q.device or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 (B, Hq, Sq) tensor on q's device")
    sq, sk, sv, so = q.stride(), k.stride(), v.stride(), out.stride()
    st = _LL12(sq[0], sq[1], sq[2], sk[0], sk[1], sk[2], sv[0], sv[1], sv[2], so[0], so[1], so[2])
    a = ctypes.addressof(st)   # `st` stays alive until the call returns
    dev = q.get_device()
    rc = _call_on(dev, lambda: lib().fa_fwd_strided(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr() if lse is not None else None,
        B, Sq, Sk, Hq, Hkv, D, a, a + 24, a + 48, a + 72, float(scale), int(bool(causal)), code,
        _stream_handle(stream, dev)))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd")
    return out, lse


fa_fwd_strided = fa_fwd


def fa_merge(o_parts, lse_parts, *, out=None, lse=None, return_lse=True, stream=None):
    """Merge partial attention results over disjoint key sets.

    o_parts: (n, B, Sq, Hq, D) contiguous 16-bit CUDA tensor; lse_parts:
    (n, B, Hq, Sq) contiguous float32. Returns (O, LSE) like fa_fwd.
    """
    import torch

    if o_parts.dim() != 5 or lse_parts.dim() != 4:
        raise ValueError("o_parts must be (n, B, Sq, Hq, D) and lse_parts (n, B, Hq, Sq)")
    n, B, Sq, Hq, D = o_parts.shape
    if tuple(lse_parts.shape) != (n, B, Hq, Sq) or lse_parts.dtype != torch.float32:
        raise ValueError("lse_parts must be float32 (n, B, Hq, Sq)")
    if not (o_parts.is_cuda and lse_parts.is_cuda and o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous CUDA tensors")
    if lse_parts.device != o_parts.device:
        raise ValueError("o_parts and lse_parts must be on one device")
    code = _dtype_code(o_parts)
    if out is None:
        out = torch.empty((B, Sq, Hq, D), dtype=o_parts.dtype, device=o_parts.device)
    else:
        _check_result("out", out, (B, Sq, Hq, D), o_parts.dtype, o_parts.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=o_parts.device)
    elif lse is not None:
        _check_result("lse", lse, (B, Hq, Sq), torch.float32, o_parts.device)
    with torch.cuda.device(o_parts.device):
        rc = lib().fa_merge(o_parts.data_ptr(), lse_parts.data_ptr(), n, out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, Sq, Hq, D, code,
                            _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_merge")
    return out, lse


def fa_decode_workspace_size(B, Sq, Sk, Hq, Hkv, D, num_splits=0) -> int:
    """Workspace bytes fa_fwd_decode needs on the current device."""
    out = ctypes.c_ulonglong(0)
    rc = lib().fa_decode_workspace_size(B, Sq, Sk, Hq, Hkv, D, num_splits, ctypes.byref(out))
    if rc != FA_OK:
        raise FAError(rc, "fa_decode_workspace_size")
    return int(out.value)


def fa_fwd_decode(q, k, v, *, scale=None, causal=False, num_splits=0, workspace=None, out=None, lse=None,
                  return_lse=True, stream=None):
    """Split-KV attention for few query rows per KV head (decode).

    Same tensors and result as fa_fwd (contiguous (B, S, H, D)); requires
    (Hq / Hkv) * Sq <= 128. ``workspace`` is a CUDA uint8 tensor of at least
    fa_decode_workspace_size(...) bytes; when omitted one is allocated here
    (through torch's allocator) for this call.
    """
    import torch

    _check_qkv_device(q, k, v)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        need = fa_decode_workspace_size(B, Sq, Sk, Hq, Hkv, D, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        elif workspace is not None:
            _check_workspace(workspace, q.device)   # its size is checked by the C call
        if out is None:
            out = torch.empty_like(q)
        else:
            _check_result("out", out, q.shape, q.dtype, q.device)
        if lse is None and return_lse:
            lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
        elif lse is not None:
            _check_result("lse", lse, (B, Hq, Sq), torch.float32, q.device)
        rc = lib().fa_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, Sq, Sk, Hq, Hkv, D, float(scale),
                                 int(bool(causal)), code, int(num_splits),
                                 workspace.data_ptr() if workspace is not None else None,
                                 workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                 _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_decode")
    return out, lse


def fa_fwd_decode_noalloc(q, k, v, *, scale=None, causal=False, num_splits=0, out=None, lse=None,
                          return_lse=True, stream=None):
    """fa_fwd_decode whose split workspace is the library's fixed 16 MiB
    device array, for callers that cannot allocate device memory when they
    call (see include/fa.h). Calls that overlap on the GPU share that array
    and race; order them on one stream."""
    import torch

    _check_qkv_device(q, k, v)
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_result("out", out, q.shape, q.dtype, q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    elif lse is not None:
        _check_result("lse", lse, (B, Hq, Sq), torch.float32, q.device)
    with torch.cuda.device(q.device):
        rc = lib().fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                         lse.data_ptr() if lse is not None else None, B, Sq, Sk, Hq, Hkv, D,
                                         float(scale), int(bool(causal)), code, int(num_splits),
                                         _stream_handle(stream))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_decode_noalloc")
    return out, lse


def fa_decode_splits(B, Sq, Sk, Hq, Hkv, D, num_splits=0, num_sms=152) -> int:
    """Key ranges fa_fwd_decode would use on a GPU with ``num_sms`` SMs (host only)."""
    out = ctypes.c_int(0)
    rc = lib().fa_decode_splits(B, Sq, Sk, Hq, Hkv, D, num_splits, num_sms, ctypes.byref(out))
    if rc != FA_OK:
        raise FAError(rc, "fa_decode_splits")
    return int(out.value)


def fa_fwd_host_workspace_size(B, Sq, Sk, Hq, Hkv, D) -> int:
    """Device bytes fa_fwd_host needs (a device copy of q, k, v, O and LSE)."""
    out = ctypes.c_ulonglong(0)
    rc = lib().fa_fwd_host_workspace_size(B, Sq, Sk, Hq, Hkv, D, ctypes.byref(out))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_host_workspace_size")
    return int(out.value)


def fa_fwd_host(q, k, v, *, scale=None, causal=False, out=None, lse=None, return_lse=True, workspace=None,
                device=None, stream=None, synchronize=True):
    """Attention on tensors in host memory: copies in, kernel and copies out
    pipelined per chunk of batches or KV heads (include/fa.h, fa_fwd_host).

    q: (B, Sq, Hq, D); k, v: (B, Sk, Hkv, D) contiguous CPU tensors of one
    16-bit dtype (page-locked memory lets the copies overlap the kernels).
    ``out``/``lse`` are CPU tensors to fill (allocated page-locked when
    omitted). ``workspace`` is a CUDA uint8 tensor of at least
    fa_fwd_host_workspace_size(...) bytes (allocated for this call when
    omitted). With ``synchronize`` the call returns once the results are in
    ``out``/``lse``; otherwise the caller synchronises ``stream`` first.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D CPU tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k and v must share one dtype")
    B, Sq, Hq, D = q.shape
    Bk, Sk, Hkv, Dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or Dk != D:
        raise ValueError("k and v must be (B, Sk, Hkv, D) matching q")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    elif tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype or out.is_cuda or not out.is_contiguous():
        raise ValueError("out must be a contiguous CPU tensor shaped and typed like q")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, pin_memory=True)
    elif lse is not None and (tuple(lse.shape) != (B, Hq, Sq) or lse.dtype != torch.float32 or lse.is_cuda
                              or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 (B, Hq, Sq) CPU tensor")
    dev = torch.cuda.current_device() if device is None else torch.device(device).index
    need = fa_fwd_host_workspace_size(B, Sq, Sk, Hq, Hkv, D)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=torch.device("cuda", dev))
    elif (not workspace.is_cuda or workspace.get_device() != dev or not workspace.is_contiguous()
          or workspace.numel() * workspace.element_size() < need):
        raise ValueError(f"workspace must be a contiguous CUDA tensor of at least {need} bytes on cuda:{dev}")

    def call():
        h = _stream_handle(stream, dev)
        rc = lib().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr() if lse is not None else None, B, Sq, Sk, Hq, Hkv, D, float(scale),
                               int(bool(causal)), code, workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), h)
        if rc != FA_OK:
            raise FAError(rc, "fa_fwd_host")
        if synchronize:
            (stream if stream is not None else torch.cuda.current_stream(dev)).synchronize()

    _call_on(dev, call)
    return out, lse


def fa_fwd_host_plan(B, Sq, Sk, Hq, Hkv, D, causal):
    """fa_fwd_host's chunks for these sizes (host only): an (n, 9) int32 array
    of rows (b0, b1, h0, h1, r0, r1, k0, k1, lim)."""
    import numpy as np

    n = ctypes.c_int(0)
    args = (int(B), int(Sq), int(Sk), int(Hq), int(Hkv), int(D), int(causal))
    rc = lib().fa_fwd_host_plan(*args, None, 0, ctypes.byref(n))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_host_plan")
    out = np.zeros((n.value, 9), dtype=np.int32)
    rc = lib().fa_fwd_host_plan(*args, out.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_host_plan")
    return out


def fa_status(stream=None) -> int:
    """Synchronise the stream; return and clear the device status word."""
    return int(lib().fa_status(_stream_handle(stream)))


def fa_status_string(code: int) -> str:
    return lib().fa_status_string(int(code)).decode()


def fa_version() -> int:
    return int(lib().fa_version())


def fa_debug_set_fault(skip_load: int, timeout_ms: int = 0) -> int:
    """Test hook: drop K/V load ``skip_load`` of every CTA (-1 = off)."""
    return int(lib().fa_debug_set_fault(int(skip_load), int(timeout_ms)))


def fa_fwd_schedule(B: int, Sq: int, Sk: int, Hq: int, Hkv: int, causal: bool, num_sms: int) -> int:
    """1 if fa_fwd would run key-split items for these sizes, 0 for row-tile pairs (host only)."""
    out = ctypes.c_int(-1)
    rc = lib().fa_fwd_schedule(int(B), int(Sq), int(Sk), int(Hq), int(Hkv), int(causal), int(num_sms),
                               ctypes.byref(out))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_schedule")
    return int(out.value)


def fa_fwd_work_items(B: int, Sq: int, Sk: int, Hq: int, Hkv: int, causal: bool, key_split: int, num_sms: int):
    """The persistent kernel's work items for these sizes (host only): an
    (n_items, 8) int32 array of rows (b, hq0, hq1, kvh, r0, r1, n_kv, cta),
    and the CTA count."""
    import numpy as np

    n = ctypes.c_int(0)
    g = ctypes.c_int(0)
    rc = lib().fa_fwd_work_items(int(B), int(Sq), int(Sk), int(Hq), int(Hkv), int(causal), int(key_split),
                                 int(num_sms), None, 0, ctypes.byref(n), ctypes.byref(g))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_work_items")
    items = np.zeros((n.value, 8), dtype=np.int32)
    rc = lib().fa_fwd_work_items(int(B), int(Sq), int(Sk), int(Hq), int(Hkv), int(causal), int(key_split),
                                 int(num_sms), items.ctypes.data_as(ctypes.c_void_p), n.value, ctypes.byref(n),
                                 ctypes.byref(g))
    if rc != FA_OK:
        raise FAError(rc, "fa_fwd_work_items")
    return items, int(g.value)


def fa_debug_set_schedule(mode: int) -> int:
    """Test hook: -1 cost model (default), 0 row-tile pairs, 1 key-split items."""
    return int(lib().fa_debug_set_schedule(int(mode)))
