"""ctypes binding of the C ABI in ``include/etattn.h``.

The functions ``attn_fwd``, ``attn_fwd_ex``, ``attn_bwd``, ``attn_bwd_workspace_size``,
``attn_fwd_splitkv``, ``attn_fwd_splitkv_noalloc``,
``attn_fwd_splitkv_workspace_size``, ``attn_fwd_splitkv_plan``,
``attn_fwd_global``,
``attn_fwd_varlen_splitkv``, ``attn_fwd_varlen_splitkv_workspace_size``,
``attn_fwd_varlen_splitkv_plan``,
``attn_fwd_varlen_global``,
``attn_fwd_varlen``, ``attn_fwd_varlen_ex``, ``attn_fwd_host``, ``attn_fwd_varlen_host``,
``attn_fwd_varlen_host_plan``,
``etattn_status_string``, ``etattn_last_cuda_error``,
``etattn_read_device_status``, ``etattn_selftest_wait_timeout`` and
``etattn_version`` have the C names and
arguments (pointers as ints).  The helpers ``attention`` and
``attention_varlen`` marshal torch CUDA tensors (output allocation, strides,
the current stream) and call them; every step of the computation runs in the
library's kernels.  There is no fallback: if the
library is missing or cannot be loaded, an error is raised.
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libetattn.so")

ETATTN_F16 = 0
ETATTN_BF16 = 1
STATUS_NAMES = {
    0: "ETATTN_OK", 1: "ETATTN_ERR_NULL_PTR", 2: "ETATTN_ERR_BAD_DTYPE", 3: "ETATTN_ERR_BAD_SHAPE",
    4: "ETATTN_ERR_BAD_HEADS", 5: "ETATTN_ERR_BAD_STRIDE", 6: "ETATTN_ERR_BAD_ALIGN", 7: "ETATTN_ERR_ALIAS",
    8: "ETATTN_ERR_BAD_SCALE", 9: "ETATTN_ERR_BAD_SEQLENS", 10: "ETATTN_ERR_LAUNCH", 11: "ETATTN_ERR_DEVICE",
    12: "ETATTN_ERR_NO_DEVICE",
}
globals().update({name: code for code, name in STATUS_NAMES.items()})


class EtattnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {STATUS_NAMES.get(code, code)} ({etattn_status_string(code)})"
        if code == 10:
            msg += f"; cudaError={etattn_last_cuda_error()}"
        super().__init__(msg)


_lib = None
_lock = threading.Lock()
_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_int = ctypes.c_int


def load_library(path: str | None = None):
    """Load libetattn.so (building it first when it is absent and nvcc is
    available).  Raises OSError / RuntimeError when it cannot be loaded."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            from . import build_lib
            path = build_lib.build()
        lib = ctypes.CDLL(path)
        lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _i64p, _int,
                                 ctypes.c_float, _vp]
        lib.attn_fwd.restype = _int
        lib.attn_fwd_ex.argtypes = [_vp] * 5 + [_int] * 7 + [_i64p] + [_int] * 3 + [ctypes.c_float, _vp]
        lib.attn_fwd_ex.restype = _int
        lib.attn_fwd_varlen_ex.argtypes = [_vp] * 9 + [_int] * 9 + [_i64p] + [_int] * 3 + [ctypes.c_float, _vp]
        lib.attn_fwd_varlen_ex.restype = _int
        lib.attn_fwd_varlen_splitkv.argtypes = ([_vp] * 9 + [_int] * 9 + [_i64p] + [_int] * 3 +
                                                [ctypes.c_float, _int, _vp, ctypes.c_size_t, _vp])
        lib.attn_fwd_varlen_splitkv.restype = _int
        lib.attn_fwd_varlen_splitkv_plan.argtypes = [_int] * 5 + [ctypes.POINTER(_int)]
        lib.attn_fwd_varlen_splitkv_plan.restype = _int
        lib.attn_fwd_varlen_splitkv_workspace_size.argtypes = [_int] * 4
        lib.attn_fwd_varlen_splitkv_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_varlen_global.argtypes = [_vp] * 9 + [_int] * 9 + [_i64p] + [_int] * 4 + [ctypes.c_float, _vp]
        lib.attn_fwd_varlen_global.restype = _int
        lib.attn_fwd_splitkv.argtypes = ([_vp] * 5 + [_int] * 7 + [_i64p] + [_int] * 3 + [ctypes.c_float, _int, _vp,
                                         ctypes.c_size_t, _vp])
        lib.attn_fwd_splitkv.restype = _int
        lib.attn_bwd.argtypes = [_vp] * 9 + [_int] * 7 + [_i64p] + [_int] * 3 + [ctypes.c_float, _vp, ctypes.c_size_t,
                                                                                   _vp]
        lib.attn_bwd.restype = _int
        lib.attn_bwd_workspace_size.argtypes = [_int] * 4
        lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_splitkv_noalloc.argtypes = ([_vp] * 5 + [_int] * 7 + [_i64p] + [_int] * 3 +
                                                 [ctypes.c_float, _int, _vp])
        lib.attn_fwd_splitkv_noalloc.restype = _int
        lib.attn_fwd_splitkv_workspace_size.argtypes = [_int] * 5
        lib.attn_fwd_splitkv_workspace_size.restype = ctypes.c_size_t
        lib.attn_fwd_splitkv_plan.argtypes = [_int] * 5 + [ctypes.POINTER(_int)]
        lib.attn_fwd_splitkv_plan.restype = _int
        lib.attn_fwd_global.argtypes = [_vp] * 5 + [_int] * 7 + [_i64p] + [_int] * 4 + [ctypes.c_float, _vp]
        lib.attn_fwd_global.restype = _int
        lib.attn_fwd_varlen.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _int,
                                        _int, _i64p, _int, ctypes.c_float, _vp]
        lib.attn_fwd_varlen.restype = _int
        lib.attn_fwd_host.argtypes = [_vp] * 10 + [_int] * 7 + [ctypes.c_float, _vp]
        lib.attn_fwd_host.restype = _int
        lib.attn_fwd_varlen_host.argtypes = [_vp] * 12 + [_int] * 8 + [ctypes.c_float, _vp]
        lib.attn_fwd_varlen_host.restype = _int
        lib.attn_fwd_varlen_host_plan.argtypes = [_vp, _int, _int, ctypes.POINTER(ctypes.c_int32)]
        lib.attn_fwd_varlen_host_plan.restype = _int
        lib.etattn_status_string.argtypes = [_int]
        lib.etattn_status_string.restype = ctypes.c_char_p
        lib.etattn_last_cuda_error.argtypes = []
        lib.etattn_last_cuda_error.restype = _int
        lib.etattn_read_device_status.argtypes = [ctypes.POINTER(_int), _int, _vp]
        lib.etattn_read_device_status.restype = _int
        lib.etattn_version.argtypes = []
        lib.etattn_version.restype = _int
        lib.etattn_selftest_wait_timeout.argtypes = [_int, _vp]
        lib.etattn_selftest_wait_timeout.restype = _int
        _lib = lib
        return lib


# ---------------------------------------------------------------- raw C entry points

def _strides_arg(strides):
    arr = (ctypes.c_int64 * len(strides))(*[int(s) for s in strides])
    return arr


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, D, dtype, strides, causal, scale, stream):
    """C ``attn_fwd``: pointers as ints (0 for NULL), ``strides`` 16 ints."""
    lib = load_library()
    return lib.attn_fwd(q or None, k or None, v or None, o or None, lse or None, B, Hq, Hkv, N, D, dtype,
                        _strides_arg(strides), causal, scale, stream or None)


def attn_fwd_ex(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                stream):
    """C ``attn_fwd_ex``: pointers as ints (0 for NULL), ``strides`` 16 ints."""
    lib = load_library()
    return lib.attn_fwd_ex(q or None, k or None, v or None, o or None, lse or None, B, Hq, Hkv, Nq, Nk, D, dtype,
                           _strides_arg(strides), causal, window_left, window_right, scale, stream or None)


def attn_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right, scale,
                     num_splits, workspace, workspace_bytes, stream):
    """C ``attn_fwd_splitkv``: pointers as ints (0 for NULL), ``strides`` 16 ints."""
    lib = load_library()
    return lib.attn_fwd_splitkv(q or None, k or None, v or None, o or None, lse or None, B, Hq, Hkv, Nq, Nk, D,
                                dtype, _strides_arg(strides), causal, window_left, window_right, scale, num_splits,
                                workspace or None, workspace_bytes, stream or None)


def attn_fwd_global(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left, window_right,
                    num_global, scale, stream):
    """C ``attn_fwd_global``: pointers as ints (0 for NULL), ``strides`` 16 ints."""
    lib = load_library()
    return lib.attn_fwd_global(q or None, k or None, v or None, o or None, lse or None, B, Hq, Hkv, Nq, Nk, D, dtype,
                               _strides_arg(strides), causal, window_left, window_right, num_global, scale,
                               stream or None)


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left,
             window_right, scale, workspace, workspace_bytes, stream):
    """C ``attn_bwd``: pointers as ints (0 for NULL), ``strides`` 32 ints."""
    lib = load_library()
    return lib.attn_bwd(q or None, k or None, v or None, o or None, lse or None, dout or None, dq or None, dk or None,
                        dv or None, B, Hq, Hkv, Nq, Nk, D, dtype, _strides_arg(strides), causal, window_left,
                        window_right, scale, workspace or None, workspace_bytes, stream or None)


def attn_bwd_workspace_size(B, Hq, Nq, D) -> int:
    return load_library().attn_bwd_workspace_size(B, Hq, Nq, D)


def attn_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, dtype, strides, causal, window_left,
                             window_right, scale, num_splits, stream):
    """C ``attn_fwd_splitkv_noalloc``: the split-KV call on the library's
    fixed 16 MiB scratch (no workspace argument)."""
    lib = load_library()
    return lib.attn_fwd_splitkv_noalloc(q or None, k or None, v or None, o or None, lse or None, B, Hq, Hkv, Nq, Nk,
                                        D, dtype, _strides_arg(strides), causal, window_left, window_right, scale,
                                        num_splits, stream or None)


def attn_fwd_splitkv_workspace_size(B, Hq, Nq, D, num_splits) -> int:
    return load_library().attn_fwd_splitkv_workspace_size(B, Hq, Nq, D, num_splits)


def attn_fwd_splitkv_plan(B, Hq, Hkv, Nq, Nk):
    """(status, num_splits) for the current device."""
    out = _int(0)
    rc = load_library().attn_fwd_splitkv_plan(B, Hq, Hkv, Nq, Nk, ctypes.byref(out))
    return rc, out.value


def attn_fwd_varlen_ex(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host, num_seqs,
                       max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal, window_left,
                       window_right, scale, stream):
    """C ``attn_fwd_varlen_ex``: pointers (device offsets and optional host
    mirrors) as ints; ``strides`` 12 ints."""
    lib = load_library()
    return lib.attn_fwd_varlen_ex(q or None, k or None, v or None, o or None, lse or None, cu_seqlens_q or None,
                                  cu_seqlens_k or None, cu_seqlens_q_host or None, cu_seqlens_k_host or None,
                                  num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype,
                                  _strides_arg(strides), causal, window_left, window_right, scale, stream or None)


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, cu_seqlens_host, num_seqs, max_seqlen, total_tokens, Hq, Hkv, D,
                    dtype, strides, causal, scale, stream):
    """C ``attn_fwd_varlen``: pointers as ints; ``cu_seqlens_host`` is an int
    address of a host int32 array or 0; ``strides`` 12 ints."""
    lib = load_library()
    return lib.attn_fwd_varlen(q or None, k or None, v or None, o or None, lse or None, cu_seqlens or None,
                               cu_seqlens_host or None, num_seqs, max_seqlen, total_tokens, Hq, Hkv, D, dtype,
                               _strides_arg(strides), causal, scale, stream or None)


def attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev, o_dev, lse_dev, B, Hq, Hkv, N, D,
                  dtype, causal, scale, stream):
    """C ``attn_fwd_host``: host and device buffer addresses as ints."""
    lib = load_library()
    return lib.attn_fwd_host(q_host or None, k_host or None, v_host or None, o_host or None, lse_host or None,
                             q_dev or None, k_dev or None, v_dev or None, o_dev or None, lse_dev or None, B, Hq,
                             Hkv, N, D, dtype, causal, scale, stream or None)


def attn_fwd_varlen_host_plan(cu_seqlens, max_chunks=8):
    """C ``attn_fwd_varlen_host_plan`` on a host sequence of offsets: (status
    or chunk count k, the k + 1 run bounds)."""
    cu = (ctypes.c_int32 * max(len(cu_seqlens), 1))(*[int(x) for x in cu_seqlens])
    bounds = (ctypes.c_int32 * 9)()
    k = load_library().attn_fwd_varlen_host_plan(ctypes.addressof(cu), len(cu_seqlens) - 1, max_chunks, bounds)
    return k, list(bounds[:k + 1]) if k > 0 else []


def attn_fwd_varlen_host(q_host, k_host, v_host, o_host, lse_host, cu_seqlens_host, q_dev, k_dev, v_dev, o_dev,
                         lse_dev, cu_seqlens_dev, num_seqs, max_seqlen, total_tokens, Hq, Hkv, D, dtype, causal,
                         scale, stream):
    """C ``attn_fwd_varlen_host``: host and device buffer addresses as ints."""
    lib = load_library()
    return lib.attn_fwd_varlen_host(q_host or None, k_host or None, v_host or None, o_host or None,
                                    lse_host or None, cu_seqlens_host or None, q_dev or None, k_dev or None,
                                    v_dev or None, o_dev or None, lse_dev or None, cu_seqlens_dev or None,
                                    num_seqs, max_seqlen, total_tokens, Hq, Hkv, D, dtype, causal, scale,
                                    stream or None)


def etattn_status_string(code: int) -> str:
    return load_library().etattn_status_string(code).decode()


def etattn_last_cuda_error() -> int:
    return load_library().etattn_last_cuda_error()


def etattn_read_device_status(clear: bool = True, stream: int = 0) -> int:
    out = _int(0)
    rc = load_library().etattn_read_device_status(ctypes.byref(out), 1 if clear else 0, stream or None)
    if rc != 0:
        raise EtattnError(rc, "etattn_read_device_status")
    return out.value


def etattn_version() -> int:
    return load_library().etattn_version()


def etattn_selftest_wait_timeout(limit_us: int, stream: int = 0) -> int:
    """C ``etattn_selftest_wait_timeout``: enqueue the bounded-wait self-test
    (a wait of limit_us microseconds that runs out and sets the device status
    word).  Returns the status code."""
    return load_library().etattn_selftest_wait_timeout(limit_us, stream or None)


# ---------------------------------------------------------------- torch marshalling

def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return ETATTN_F16
    if t.dtype == torch.bfloat16:
        return ETATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float16 or bfloat16")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def attention(q, k, v, *, causal: bool = True, scale: float | None = None, window_left: int = -1,
              window_right: int = -1, out=None, lse=None, return_lse: bool = True, stream=None):
    """Batched (GQA-capable) attention on CUDA tensors.

    q: [B, Hq, Nq, D]; k, v: [B, Hkv, Nk, D] (any strides with d contiguous,
    e.g. a [B, N, H, D] buffer viewed through permute).  With Nk != Nq the
    last query row aligns with the last key; ``window_left`` /
    ``window_right`` >= 0 bound the keys a row reads around its own key
    position.  Returns (o, lse) with o a new [B, Hq, Nq, D] tensor (or
    ``out``) and lse a new [B, Hq, Nq] FP32 tensor (or ``lse``; None when
    ``return_lse`` is False).  Square calls without a window go through
    ``attn_fwd``, the others through ``attn_fwd_ex``."""
    import torch
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 [B, Hq, Nq] tensor")
    strides = [*q.stride(), *k.stride(), *v.stride(), *out.stride()]
    lse_ptr = lse.data_ptr() if lse is not None else 0
    square = Nq == Nk and window_left < 0 and window_right < 0
    with torch.cuda.device(q.device):
        if square:
            rc = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv, Nq, D,
                          _dtype_code(q), strides, 1 if causal else 0, float(scale), _stream_handle(stream))
        else:
            rc = attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, B, Hq, Hkv, Nq, Nk,
                             D, _dtype_code(q), strides, 1 if causal else 0, int(window_left), int(window_right),
                             float(scale), _stream_handle(stream))
    if rc != 0:
        raise EtattnError(rc, "attn_fwd" if square else "attn_fwd_ex")
    return out, lse


def attention_splitkv(q, k, v, *, causal: bool = True, scale: float | None = None, window_left: int = -1,
                      window_right: int = -1, num_splits: int | None = None, workspace=None, out=None, lse=None,
                      return_lse: bool = True, stream=None):
    """``attention`` computed with the keys cut into ``num_splits`` slices
    (default: the library's plan for the current device) and merged by a
    second launch.  ``workspace`` is a CUDA uint8 tensor of at least
    ``attn_fwd_splitkv_workspace_size`` bytes (allocated here when None)."""
    import torch
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        if num_splits is None:
            rc, num_splits = attn_fwd_splitkv_plan(B, Hq, Hkv, Nq, Nk)
            if rc != 0:
                raise EtattnError(rc, "attn_fwd_splitkv_plan")
        need = attn_fwd_splitkv_workspace_size(B, Hq, Nq, D, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if out is None:
            out = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
        if lse is None and return_lse:
            lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
        strides = [*q.stride(), *k.stride(), *v.stride(), *out.stride()]
        ws_ptr = workspace.data_ptr() if workspace is not None else 0
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr() if lse is not None else 0, B, Hq, Hkv, Nq, Nk, D, _dtype_code(q),
                              strides, 1 if causal else 0, int(window_left), int(window_right), float(scale),
                              int(num_splits), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != 0:
        raise EtattnError(rc, "attn_fwd_splitkv")
    return out, lse


def attention_global(q, k, v, *, num_global: int, causal: bool = True, scale: float | None = None,
                     window_left: int = -1, window_right: int = -1, out=None, lse=None, return_lse: bool = True,
                     stream=None):
    """``attention`` with ``num_global`` global tokens beside the window (the
    first positions read and are read by every row, under the causal mask)."""
    import torch
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        if out is None:
            out = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
        if lse is None and return_lse:
            lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
        strides = [*q.stride(), *k.stride(), *v.stride(), *out.stride()]
        rc = attn_fwd_global(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr() if lse is not None else 0, B, Hq, Hkv, Nq, Nk, D, _dtype_code(q), strides,
                             1 if causal else 0, int(window_left), int(window_right), int(num_global), float(scale),
                             _stream_handle(stream))
    if rc != 0:
        raise EtattnError(rc, "attn_fwd_global")
    return out, lse


def attention_backward(q, k, v, o, lse, dout, *, causal: bool = True, scale: float | None = None,
                       window_left: int = -1, window_right: int = -1, dq=None, dk=None, dv=None, workspace=None,
                       stream=None):
    """Gradients (dq, dk, dv) of ``attention`` for upstream gradient ``dout``,
    given the forward's output ``o`` and logsumexp ``lse`` ([B, Hq, Nq] FP32).
    Shapes and strides as for ``attention``; the outputs are allocated when
    not given, and so is the FP32 workspace (``attn_bwd_workspace_size``)."""
    import torch
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, Hq, Nq] tensor")
    with torch.cuda.device(q.device):
        if dq is None:
            dq = torch.empty((B, Hq, Nq, D), dtype=q.dtype, device=q.device)
        if dk is None:
            dk = torch.empty((B, Hkv, Nk, D), dtype=q.dtype, device=q.device)
        if dv is None:
            dv = torch.empty((B, Hkv, Nk, D), dtype=q.dtype, device=q.device)
        need = attn_bwd_workspace_size(B, Hq, Nq, D)
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        strides = [*q.stride(), *k.stride(), *v.stride(), *o.stride(), *dout.stride(), *dq.stride(), *dk.stride(),
                   *dv.stride()]
        ws_ptr = workspace.data_ptr() if workspace is not None else 0
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                      dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Nq, Nk, D, _dtype_code(q), strides,
                      1 if causal else 0, int(window_left), int(window_right), float(scale), ws_ptr, ws_bytes,
                      _stream_handle(stream))
    if rc != 0:
        raise EtattnError(rc, "attn_bwd")
    return dq, dk, dv


def attn_fwd_varlen_splitkv(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host,
                            num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal,
                            window_left, window_right, scale, num_splits, workspace, workspace_bytes, stream):
    """C ``attn_fwd_varlen_splitkv``: pointers as ints; ``strides`` 12 ints."""
    lib = load_library()
    return lib.attn_fwd_varlen_splitkv(q or None, k or None, v or None, o or None, lse or None, cu_seqlens_q or None,
                                       cu_seqlens_k or None, cu_seqlens_q_host or None, cu_seqlens_k_host or None,
                                       num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype,
                                       _strides_arg(strides), causal, window_left, window_right, scale, num_splits,
                                       workspace or None, workspace_bytes, stream or None)


def attn_fwd_varlen_splitkv_plan(num_seqs, Hq, Hkv, max_seqlen_q, max_seqlen_k):
    """(status, num_splits) for the current device."""
    out = _int(0)
    rc = load_library().attn_fwd_varlen_splitkv_plan(num_seqs, Hq, Hkv, max_seqlen_q, max_seqlen_k,
                                                      ctypes.byref(out))
    return rc, out.value


def attn_fwd_varlen_splitkv_workspace_size(total_q, Hq, D, num_splits) -> int:
    return load_library().attn_fwd_varlen_splitkv_workspace_size(total_q, Hq, D, num_splits)


def attn_fwd_varlen_global(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host,
                           num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype, strides, causal,
                           window_left, window_right, num_global, scale, stream):
    """C ``attn_fwd_varlen_global``: pointers as ints; ``strides`` 12 ints."""
    lib = load_library()
    return lib.attn_fwd_varlen_global(q or None, k or None, v or None, o or None, lse or None, cu_seqlens_q or None,
                                      cu_seqlens_k or None, cu_seqlens_q_host or None, cu_seqlens_k_host or None,
                                      num_seqs, max_seqlen_q, max_seqlen_k, total_q, total_k, Hq, Hkv, D, dtype,
                                      _strides_arg(strides), causal, window_left, window_right, num_global, scale,
                                      stream or None)


def attention_varlen(q, k, v, cu_seqlens, max_seqlen: int, *, causal: bool = True, scale: float | None = None,
                     cu_seqlens_k=None, max_seqlen_k: int | None = None, window_left: int = -1,
                     window_right: int = -1, cu_seqlens_host=None, cu_seqlens_k_host=None, out=None, lse=None,
                     return_lse: bool = True, stream=None, num_splits: int = 1, num_global: int = 0,
                     workspace=None):
    """Packed variable-length attention on CUDA tensors.

    q: [T, Hq, D]; k, v: [Tk, Hkv, D]; cu_seqlens: int32 CUDA tensor [S+1]
    of query offsets; ``cu_seqlens_k`` (default: cu_seqlens) the key
    offsets, with ``max_seqlen_k`` their longest length.  The host mirrors
    ``cu_seqlens_host`` / ``cu_seqlens_k_host`` (optional int32 CPU tensors)
    are validated before launch.  Returns (o [T, Hq, D], lse [Hq, T] FP32 or
    None).  Self-attention without a window goes through
    ``attn_fwd_varlen``, the rest through ``attn_fwd_varlen_ex``; with
    ``num_splits`` > 1 through ``attn_fwd_varlen_splitkv`` and with
    ``num_global`` > 0 through ``attn_fwd_varlen_global`` (``workspace``: the
    split-KV scratch, a CUDA uint8 tensor allocated here when None)."""
    import torch
    T, Hq, D = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    S = cu_seqlens.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    for name, t in (("cu_seqlens", cu_seqlens), ("cu_seqlens_k", cu_seqlens_k)):
        if t is not None and (t.dtype != torch.int32 or not t.is_cuda):
            raise TypeError(f"{name} must be an int32 CUDA tensor")
    if out is None:
        out = torch.empty((T, Hq, D), dtype=q.dtype, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)

    def host_addr(t):
        if t is None:
            return None, 0
        t = t.to(torch.int32).contiguous()
        return t, t.data_ptr()

    cu_host, host_ptr = host_addr(cu_seqlens_host)
    cu_k_host, host_k_ptr = host_addr(cu_seqlens_k_host)
    strides = [*q.stride(), *k.stride(), *v.stride(), *out.stride()]
    lse_ptr = lse.data_ptr() if lse is not None else 0
    plain = (cu_seqlens_k is None and cu_k_host is None and window_left < 0 and window_right < 0 and num_splits <= 1
             and num_global <= 0)
    with torch.cuda.device(q.device):
        if num_global > 0 or num_splits > 1:
            cu_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
            if cu_seqlens_k is None:
                host_k_ptr = host_ptr
            mk = int(max_seqlen if max_seqlen_k is None else max_seqlen_k)
            need = 0 if num_global > 0 else attn_fwd_varlen_splitkv_workspace_size(T, Hq, D, int(num_splits))
            if workspace is None and need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            ws_ptr = workspace.data_ptr() if workspace is not None else 0
            ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
            common = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr, cu_seqlens.data_ptr(),
                      cu_k.data_ptr(), host_ptr, host_k_ptr, S, int(max_seqlen), mk, T, Tk, Hq, Hkv, D,
                      _dtype_code(q), strides, 1 if causal else 0, int(window_left), int(window_right))
            if num_global > 0:
                rc = attn_fwd_varlen_global(*common, int(num_global), float(scale), _stream_handle(stream))
                name = "attn_fwd_varlen_global"
            else:
                rc = attn_fwd_varlen_splitkv(*common, float(scale), int(num_splits), ws_ptr, ws_bytes,
                                             _stream_handle(stream))
                name = "attn_fwd_varlen_splitkv"
        elif plain:
            rc = attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                                 cu_seqlens.data_ptr(), host_ptr, S, int(max_seqlen), T, Hq, Hkv, D, _dtype_code(q),
                                 strides, 1 if causal else 0, float(scale), _stream_handle(stream))
        else:
            cu_k = cu_seqlens if cu_seqlens_k is None else cu_seqlens_k
            if cu_seqlens_k is None:
                host_k_ptr = host_ptr
            mk = int(max_seqlen if max_seqlen_k is None else max_seqlen_k)
            rc = attn_fwd_varlen_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse_ptr,
                                    cu_seqlens.data_ptr(), cu_k.data_ptr(), host_ptr, host_k_ptr, S, int(max_seqlen),
                                    mk, T, Tk, Hq, Hkv, D, _dtype_code(q), strides, 1 if causal else 0,
                                    int(window_left), int(window_right), float(scale), _stream_handle(stream))
    del cu_host, cu_k_host
    if rc != 0:
        if num_global <= 0 and num_splits <= 1:
            name = "attn_fwd_varlen" if plain else "attn_fwd_varlen_ex"
        raise EtattnError(rc, name)
    return out, lse
