"""ctypes binding of libsdpa_gb300.so (argument marshalling only).

The functions here carry the C ABI's names and arguments; tensors are
torch.Tensors that already live on the GPU, passed by their data pointers.
Every step of the computation runs in the library's CUDA kernels; if the
library cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

SDPA_OK = 0
SDPA_ERR_INVALID_ARG = 1
SDPA_ERR_UNSUPPORTED = 2
SDPA_ERR_MISALIGNED = 3
SDPA_ERR_WORKSPACE = 4
SDPA_ERR_CUDA = 5
SDPA_ERR_TIMEOUT = 6
SDPA_BF16 = 0
SDPA_FP16 = 1
SDPA_FP8_E4M3 = 2
SDPA_MASK_NONE = 0
SDPA_MASK_CAUSAL = 1
SDPA_MASK_CAUSAL_BOTTOM_RIGHT = 2

STATUS_NAMES = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID_ARG", 2: "SDPA_ERR_UNSUPPORTED",
                3: "SDPA_ERR_MISALIGNED", 4: "SDPA_ERR_WORKSPACE", 5: "SDPA_ERR_CUDA",
                6: "SDPA_ERR_TIMEOUT"}

# Exported symbols, in the order include/sdpa.h declares them.
EXPORTS = ("sdpa_fwd", "sdpa_varlen_fwd", "sdpa_fwd_ex", "sdpa_varlen_fwd_ex", "sdpa_fwd_fp8",
           "sdpa_varlen_fwd_fp8",
           "sdpa_bwd_workspace_size", "sdpa_bwd", "sdpa_varlen_bwd_workspace_size",
           "sdpa_varlen_bwd", "sdpa_bwd_ex_workspace_size", "sdpa_varlen_bwd_ex_workspace_size",
           "sdpa_bwd_ex", "sdpa_varlen_bwd_ex", "sdpa_bwd_noalloc", "sdpa_last_error",
           "sdpa_check_device_error", "sdpa_selftest_wait_timeout", "sdpa_set_kernel_timer",
           "sdpa_set_forward_variant", "sdpa_set_backward_variant", "sdpa_last_backward_variant",
           "sdpa_set_backward_grid_limit", "sdpa_version")


class SdpaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_Z = ctypes.c_size_t

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the shared library (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if path is None:
            path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"CUDA attention library not found at {path}")
        lib = ctypes.CDLL(path)
        lib.sdpa_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]
        lib.sdpa_varlen_fwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                        _F, _I, _I, _P]
        lib.sdpa_fwd_ex.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]
        lib.sdpa_varlen_fwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                           _I, _F, _I, _I, _I, _P]
        lib.sdpa_fwd_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                     _F, _I, _I, _I, _P]
        lib.sdpa_varlen_fwd_fp8.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                            _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P]
        lib.sdpa_bwd_ex_workspace_size.argtypes = [_I, _I, _I, _I, _I]
        lib.sdpa_bwd_ex_workspace_size.restype = _Z
        lib.sdpa_varlen_bwd_ex_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.sdpa_varlen_bwd_ex_workspace_size.restype = _Z
        lib.sdpa_bwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                    _F, _I, _I, _I, _I, _P, _Z, _P]
        lib.sdpa_varlen_bwd_ex.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                           _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _I, _P, _Z, _P]
        lib.sdpa_bwd_workspace_size.argtypes = [_I, _I, _I, _I]
        lib.sdpa_bwd_workspace_size.restype = _Z
        lib.sdpa_varlen_bwd_workspace_size.argtypes = [_I, _I, _I]
        lib.sdpa_varlen_bwd_workspace_size.restype = _Z
        lib.sdpa_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                                 _I, _P, _Z, _P]
        lib.sdpa_varlen_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                        _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]
        lib.sdpa_bwd_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                         _F, _I, _I, _P]
        lib.sdpa_last_error.restype = ctypes.c_char_p
        lib.sdpa_check_device_error.argtypes = [_P]
        lib.sdpa_selftest_wait_timeout.argtypes = [_I, _P]
        lib.sdpa_selftest_wait_timeout.restype = _I
        lib.sdpa_version.restype = ctypes.c_char_p
        lib.sdpa_set_forward_variant.argtypes = [_I]
        lib.sdpa_set_forward_variant.restype = _I
        lib.sdpa_set_backward_variant.argtypes = [_I]
        lib.sdpa_set_backward_variant.restype = _I
        lib.sdpa_last_backward_variant.argtypes = []
        lib.sdpa_last_backward_variant.restype = _I
        lib.sdpa_set_backward_grid_limit.argtypes = [_I]
        lib.sdpa_set_backward_grid_limit.restype = _I
        lib.sdpa_set_kernel_timer.argtypes = [_P, _P]
        lib.sdpa_set_kernel_timer.restype = None
        for name in ("sdpa_fwd", "sdpa_varlen_fwd", "sdpa_bwd", "sdpa_varlen_bwd",
                     "sdpa_fwd_ex", "sdpa_varlen_fwd_ex", "sdpa_bwd_ex", "sdpa_varlen_bwd_ex",
                     "sdpa_fwd_fp8", "sdpa_varlen_fwd_fp8",
                     "sdpa_bwd_noalloc", "sdpa_check_device_error"):
            getattr(lib, name).restype = _I
        _lib = lib
        return lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int) -> None:
    if status != SDPA_OK:
        msg = load().sdpa_last_error().decode()
        raise SdpaError(status, msg)


def dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SDPA_BF16
    if t.dtype == torch.float16:
        return SDPA_FP16
    raise SdpaError(SDPA_ERR_UNSUPPORTED, f"dtype {t.dtype} (use bfloat16 or float16)")


def sdpa_fwd(q, k, v, o, lse, b, h, s_q, s_kv, d, attn_scale, causal, dtype, stream=None):
    _check(load().sdpa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), b, h, s_q, s_kv, d,
                           float(attn_scale), int(causal), int(dtype), _stream(stream)))


def sdpa_varlen_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                    max_seqlen_q, max_seqlen_kv, h, d, attn_scale, causal, dtype, stream=None):
    _check(load().sdpa_varlen_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                  _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), num_seqs, total_q,
                                  total_kv, max_seqlen_q, max_seqlen_kv, h, d, float(attn_scale),
                                  int(causal), int(dtype), _stream(stream)))


def sdpa_fwd_ex(q, k, v, o, lse, b, h, h_kv, s_q, s_kv, d, attn_scale, mask, window_left, dtype,
                stream=None):
    _check(load().sdpa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), b, h, h_kv, s_q, s_kv,
                              d, float(attn_scale), int(mask), int(window_left), int(dtype),
                              _stream(stream)))


def sdpa_varlen_fwd_ex(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv,
                       max_seqlen_q, max_seqlen_kv, h, h_kv, d, attn_scale, mask, window_left,
                       dtype, stream=None):
    _check(load().sdpa_varlen_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), num_seqs, total_q,
                                     total_kv, max_seqlen_q, max_seqlen_kv, h, h_kv, d,
                                     float(attn_scale), int(mask), int(window_left), int(dtype),
                                     _stream(stream)))


def sdpa_fwd_fp8(q, k, v, o, lse, descale_q, descale_k, descale_v, scale_o, amax_o, b, h, h_kv,
                 s_q, s_kv, d, attn_scale, mask, window_left, out_dtype, stream=None):
    _check(load().sdpa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(descale_q),
                               _ptr(descale_k), _ptr(descale_v), _ptr(scale_o), _ptr(amax_o), b,
                               h, h_kv, s_q, s_kv, d, float(attn_scale), int(mask),
                               int(window_left), int(out_dtype), _stream(stream)))


def sdpa_varlen_fwd_fp8(q, k, v, o, lse, descale_q, descale_k, descale_v, scale_o, amax_o,
                        cu_seqlens_q, cu_seqlens_kv, num_seqs, total_q, total_kv, max_seqlen_q,
                        max_seqlen_kv, h, h_kv, d, attn_scale, mask, window_left, out_dtype,
                        stream=None):
    _check(load().sdpa_varlen_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(descale_q), _ptr(descale_k), _ptr(descale_v),
                                      _ptr(scale_o), _ptr(amax_o), _ptr(cu_seqlens_q),
                                      _ptr(cu_seqlens_kv), num_seqs, total_q, total_kv,
                                      max_seqlen_q, max_seqlen_kv, h, h_kv, d, float(attn_scale),
                                      int(mask), int(window_left), int(out_dtype),
                                      _stream(stream)))


def sdpa_bwd_ex_workspace_size(b, h, s_q, d, deterministic=0) -> int:
    return int(load().sdpa_bwd_ex_workspace_size(b, h, s_q, d, int(deterministic)))


def sdpa_varlen_bwd_ex_workspace_size(total_q, h, d, deterministic=0) -> int:
    return int(load().sdpa_varlen_bwd_ex_workspace_size(total_q, h, d, int(deterministic)))


def sdpa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, b, h, h_kv, s_q, s_kv, d, attn_scale, mask,
                window_left, deterministic, dtype, workspace, workspace_bytes, stream=None):
    _check(load().sdpa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), b, h, h_kv, s_q, s_kv, d, float(attn_scale),
                              int(mask), int(window_left), int(deterministic), int(dtype),
                              _ptr(workspace), int(workspace_bytes), _stream(stream)))


def sdpa_varlen_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, num_seqs,
                       total_q, total_kv, max_seqlen_q, max_seqlen_kv, h, h_kv, d, attn_scale,
                       mask, window_left, deterministic, dtype, workspace, workspace_bytes,
                       stream=None):
    _check(load().sdpa_varlen_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q),
                                     _ptr(cu_seqlens_kv), num_seqs, total_q, total_kv,
                                     max_seqlen_q, max_seqlen_kv, h, h_kv, d, float(attn_scale),
                                     int(mask), int(window_left), int(deterministic), int(dtype),
                                     _ptr(workspace), int(workspace_bytes), _stream(stream)))


def sdpa_bwd_workspace_size(b, h, s_q, d) -> int:
    return int(load().sdpa_bwd_workspace_size(b, h, s_q, d))


def sdpa_varlen_bwd_workspace_size(total_q, h, d) -> int:
    return int(load().sdpa_varlen_bwd_workspace_size(total_q, h, d))


def sdpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, s_q, s_kv, d, attn_scale, causal, dtype,
             workspace, workspace_bytes, stream=None):
    _check(load().sdpa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                           _ptr(dk), _ptr(dv), b, h, s_q, s_kv, d, float(attn_scale), int(causal),
                           int(dtype), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def sdpa_varlen_bwd(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_kv, num_seqs,
                    total_q, total_kv, max_seqlen_q, max_seqlen_kv, h, d, attn_scale, causal,
                    dtype, workspace, workspace_bytes, stream=None):
    _check(load().sdpa_varlen_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q),
                                  _ptr(cu_seqlens_kv), num_seqs, total_q, total_kv, max_seqlen_q,
                                  max_seqlen_kv, h, d, float(attn_scale), int(causal), int(dtype),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream)))


def sdpa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, b, h, s_q, s_kv, d, attn_scale, causal,
                     dtype, stream=None):
    """Dense backward without a workspace (the library's built-in scratch array)."""
    _check(load().sdpa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), b, h, s_q, s_kv, d,
                                   float(attn_scale), int(causal), int(dtype), _stream(stream)))


def sdpa_last_error() -> str:
    return load().sdpa_last_error().decode()


def sdpa_check_device_error(stream=None) -> None:
    _check(load().sdpa_check_device_error(_stream(stream)))


def sdpa_selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test (see include/sdpa.h)."""
    _check(load().sdpa_selftest_wait_timeout(int(limit_us), _stream(stream)))


def sdpa_set_kernel_timer(start_event=None, stop_event=None) -> None:
    """Record torch.cuda.Event pairs around the main kernel of later calls on this thread."""
    def handle(ev):
        if ev is None:
            return None
        if not ev.cuda_event:  # torch creates the CUDA event lazily
            ev.record()
        return ev.cuda_event
    load().sdpa_set_kernel_timer(handle(start_event), handle(stop_event))


def sdpa_set_forward_variant(variant: int) -> None:
    """0: automatic forward kernel choice, 1: one-tile kernel, 2: two-tile kernel."""
    _check(load().sdpa_set_forward_variant(int(variant)))


def sdpa_set_backward_variant(variant: int) -> None:
    """0: automatic backward main-kernel choice, 1: one CTA per key tile, 2: persistent."""
    _check(load().sdpa_set_backward_variant(int(variant)))


def sdpa_last_backward_variant() -> int:
    """Main kernel of this thread's last backward call: 1 one CTA per key tile, 2 persistent."""
    return int(load().sdpa_last_backward_variant())


def sdpa_set_backward_grid_limit(max_ctas: int) -> None:
    """Most CTAs of the persistent backward kernel on this thread (0: one per SM)."""
    _check(load().sdpa_set_backward_grid_limit(int(max_ctas)))


def sdpa_version() -> str:
    return load().sdpa_version().decode()
