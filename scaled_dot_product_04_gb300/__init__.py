"""GB300-native fused scaled-dot-product attention.

``O = softmax(attn_scale * Q K^T + causal mask) V`` plus the per-row
log-sum-exp, dense BHSD or packed THD, and its backward, computed by
hand-written sm_103a kernels behind the C ABI in ``include/sdpa.h``.

This package is the thin Python side: ``_lib`` mirrors the C entry points
one to one, and the helpers below allocate outputs with torch and call them.
PyTorch only provides device memory and streams.
"""
from __future__ import annotations

import math

from ._lib import (SDPA_BF16, SDPA_FP16, SDPA_FP8_E4M3, sdpa_fwd_fp8, sdpa_varlen_fwd_fp8,  # noqa: F401
                   SDPA_MASK_CAUSAL, SDPA_MASK_CAUSAL_BOTTOM_RIGHT,
                   SDPA_MASK_NONE, SdpaError, dtype_code, load, sdpa_bwd, sdpa_bwd_ex,
                   sdpa_bwd_ex_workspace_size, sdpa_bwd_noalloc, sdpa_bwd_workspace_size,
                   sdpa_check_device_error, sdpa_fwd, sdpa_fwd_ex, sdpa_last_error,
                   sdpa_selftest_wait_timeout,
                   sdpa_last_backward_variant, sdpa_set_backward_grid_limit,
                   sdpa_set_backward_variant,
                   sdpa_set_forward_variant, sdpa_set_kernel_timer, sdpa_varlen_bwd,
                   sdpa_varlen_bwd_ex, sdpa_varlen_bwd_ex_workspace_size,
                   sdpa_varlen_bwd_workspace_size, sdpa_varlen_fwd, sdpa_varlen_fwd_ex, sdpa_version)

__all__ = ["attention", "attention_varlen", "attention_bwd", "attention_varlen_bwd",
           "sdpa_fwd", "sdpa_varlen_fwd", "sdpa_bwd", "sdpa_varlen_bwd", "sdpa_bwd_noalloc",
           "sdpa_fwd_ex", "sdpa_varlen_fwd_ex", "sdpa_bwd_ex", "sdpa_varlen_bwd_ex",
           "sdpa_bwd_workspace_size", "sdpa_varlen_bwd_workspace_size",
           "sdpa_bwd_ex_workspace_size", "sdpa_varlen_bwd_ex_workspace_size", "sdpa_last_error",
           "sdpa_check_device_error", "sdpa_selftest_wait_timeout", "sdpa_set_forward_variant",
           "sdpa_set_backward_variant", "sdpa_last_backward_variant",
           "sdpa_set_backward_grid_limit", "sdpa_set_kernel_timer",
           "sdpa_version", "SdpaError", "load", "SDPA_MASK_NONE", "SDPA_MASK_CAUSAL",
           "SDPA_MASK_CAUSAL_BOTTOM_RIGHT", "SDPA_FP8_E4M3", "sdpa_fwd_fp8", "sdpa_varlen_fwd_fp8",
           "attention_fp8"]

_MASK_NAMES = {"none": SDPA_MASK_NONE, "top_left": SDPA_MASK_CAUSAL,
               "bottom_right": SDPA_MASK_CAUSAL_BOTTOM_RIGHT}


def _mask_code(causal, mask) -> int:
    """`mask` (an SDPA_MASK_* value or "none" / "top_left" / "bottom_right")
    overrides the plain `causal` flag when given."""
    if mask is None:
        return SDPA_MASK_CAUSAL if causal else SDPA_MASK_NONE
    return _MASK_NAMES[mask] if isinstance(mask, str) else int(mask)


def _default_scale(d: int, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def attention(q, k, v, *, scale=None, causal=False, mask=None, window_left=-1, stream=None):
    """Dense forward. q [b,h,s_q,d], k/v [b,h_kv,s_kv,d] (CUDA, contiguous) -> (o, lse).

    h_kv may divide h (grouped key/value heads); `mask` and `window_left`
    select the masks of include/sdpa.h (sdpa_mask)."""
    import torch
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    m = _mask_code(causal, mask)
    o = torch.empty_like(q)
    lse = torch.empty((b, h, s_q), dtype=torch.float32, device=q.device)
    if h_kv == h and window_left < 0 and m != SDPA_MASK_CAUSAL_BOTTOM_RIGHT:
        sdpa_fwd(q, k, v, o, lse, b, h, s_q, s_kv, d, _default_scale(d, scale), m,
                 dtype_code(q), stream)
    else:
        sdpa_fwd_ex(q, k, v, o, lse, b, h, h_kv, s_q, s_kv, d, _default_scale(d, scale), m,
                    window_left, dtype_code(q), stream)
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q, max_seqlen_kv, *,
                     scale=None, causal=False, mask=None, window_left=-1, stream=None,
                     total_q=None, total_kv=None):
    """Packed forward. q [Tq,h,d], k/v [Tkv,h_kv,d], cu_seqlens int32 on the device.

    ``total_q``/``total_kv`` default to the tensors' first dimension; pass them
    when the buffers hold spare capacity past the packed total.
    """
    import torch
    tq = q.shape[0] if total_q is None else int(total_q)
    tkv = k.shape[0] if total_kv is None else int(total_kv)
    _, h, d = q.shape
    h_kv = k.shape[1]
    m = _mask_code(causal, mask)
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[0], h), dtype=torch.float32, device=q.device)
    args = (cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q.numel() - 1, tq, tkv, int(max_seqlen_q),
            int(max_seqlen_kv))
    if h_kv == h and window_left < 0 and m != SDPA_MASK_CAUSAL_BOTTOM_RIGHT:
        sdpa_varlen_fwd(q, k, v, o, lse, *args, h, d, _default_scale(d, scale), m, dtype_code(q),
                        stream)
    else:
        sdpa_varlen_fwd_ex(q, k, v, o, lse, *args, h, h_kv, d, _default_scale(d, scale), m,
                           window_left, dtype_code(q), stream)
    return o, lse


def attention_bwd(q, k, v, o, dout, lse, *, scale=None, causal=False, mask=None, window_left=-1,
                  deterministic=False, stream=None, workspace=None):
    """Dense backward -> (dq, dk, dv).  Allocates the workspace unless one is given."""
    import torch
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    m = _mask_code(causal, mask)
    plain = (h_kv == h and window_left < 0 and m != SDPA_MASK_CAUSAL_BOTTOM_RIGHT
             and not deterministic)
    ws_bytes = (sdpa_bwd_workspace_size(b, h, s_q, d) if plain
                else sdpa_bwd_ex_workspace_size(b, h, s_q, d, int(bool(deterministic))))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if plain:
        sdpa_bwd(q, k, v, o, dout, lse, dq, dk, dv, b, h, s_q, s_kv, d, _default_scale(d, scale),
                 m, dtype_code(q), workspace, workspace.numel(), stream)
    else:
        sdpa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, b, h, h_kv, s_q, s_kv, d,
                    _default_scale(d, scale), m, window_left, int(bool(deterministic)),
                    dtype_code(q), workspace, workspace.numel(), stream)
    return dq, dk, dv


def attention_varlen_bwd(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q,
                         max_seqlen_kv, *, scale=None, causal=False, mask=None, window_left=-1,
                         deterministic=False, stream=None, workspace=None, total_q=None,
                         total_kv=None):
    """Packed backward -> (dq, dk, dv) in the packed layouts."""
    import torch
    tq = q.shape[0] if total_q is None else int(total_q)
    tkv = k.shape[0] if total_kv is None else int(total_kv)
    _, h, d = q.shape
    h_kv = k.shape[1]
    m = _mask_code(causal, mask)
    plain = (h_kv == h and window_left < 0 and m != SDPA_MASK_CAUSAL_BOTTOM_RIGHT
             and not deterministic)
    ws_bytes = (sdpa_varlen_bwd_workspace_size(tq, h, d) if plain
                else sdpa_varlen_bwd_ex_workspace_size(tq, h, d, int(bool(deterministic))))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    args = (cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q.numel() - 1, tq, tkv, int(max_seqlen_q),
            int(max_seqlen_kv))
    if plain:
        sdpa_varlen_bwd(q, k, v, o, dout, lse, dq, dk, dv, *args, h, d, _default_scale(d, scale),
                        m, dtype_code(q), workspace, workspace.numel(), stream)
    else:
        sdpa_varlen_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, *args, h, h_kv, d,
                           _default_scale(d, scale), m, window_left, int(bool(deterministic)),
                           dtype_code(q), workspace, workspace.numel(), stream)
    return dq, dk, dv


def attention_fp8(q, k, v, descale_q, descale_k, descale_v, *, scale=None, causal=False, mask=None,
                  window_left=-1, out_dtype=None, scale_o=None, want_amax=True, stream=None):
    """Dense FP8 forward.  q [b,h,s_q,d], k/v [b,h_kv,s_kv,d] as torch.float8_e4m3fn (or
    uint8 codes) on the GPU; descales are 1-element fp32 CUDA tensors.  out_dtype:
    torch.bfloat16 (default), torch.float16 or torch.float8_e4m3fn (needs scale_o).
    -> (o, lse, amax) with amax a 1-element fp32 tensor (or None)."""
    import torch
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    out_dtype = torch.bfloat16 if out_dtype is None else out_dtype
    code = {torch.bfloat16: SDPA_BF16, torch.float16: SDPA_FP16}.get(out_dtype, SDPA_FP8_E4M3)
    o = torch.empty((b, h, s_q, d), dtype=out_dtype, device=q.device)
    lse = torch.empty((b, h, s_q), dtype=torch.float32, device=q.device)
    amax = torch.empty(1, dtype=torch.float32, device=q.device) if want_amax else None
    sdpa_fwd_fp8(q, k, v, o, lse, descale_q, descale_k, descale_v, scale_o, amax, b, h, h_kv, s_q,
                 s_kv, d, _default_scale(d, scale), _mask_code(causal, mask), window_left, code,
                 stream)
    return o, lse, amax
