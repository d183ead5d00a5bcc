"""fp64 CPU oracle for scaled-dot-product attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA library: its
arithmetic lives in ``sdpa_oracle.c`` (plain C, fp64, OpenMP over independent
rows), compiled here with gcc, and this module only converts tensors to fp64
arrays and back.

Inputs are upcast exactly from their bf16/fp16 values to fp64; outputs are
fp64.  Definitions and page citations are in the header of ``sdpa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_i64 = ctypes.c_int64
_int = ctypes.c_int
_dbl = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc -O2 -fopenmp). Returns its path."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.oracle_attn_fwd_rows.argtypes = [_dp, _i64, _dp, _i64, _dp, _i64, _dp, _dp,
                                             _int, _int, _int, _dbl, _int, _ip, _int]
        lib.oracle_attn_bwd_rows.argtypes = [_dp, _i64, _dp, _i64, _dp, _i64, _dp, _i64,
                                             _dp, _dp, _dp, _int, _int, _int, _dbl, _int,
                                             _ip, _int, _ip, _int]
        lib.oracle_sdpa_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _int, _int, _int, _int, _int,
                                        _dbl, _int]
        lib.oracle_sdpa_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _int, _int, _int,
                                        _int, _int, _dbl, _int]
        lib.oracle_sdpa_varlen_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _ip, _ip, _int, _int,
                                               _int, _dbl, _int]
        lib.oracle_sdpa_varlen_bwd.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _ip,
                                               _int, _int, _int, _dbl, _int]
        lib.oracle_attn_fwd_rows_ex.argtypes = [_dp, _i64, _dp, _i64, _dp, _i64, _dp, _dp,
                                                _int, _int, _int, _dbl, _int, _int, _ip, _int]
        lib.oracle_attn_bwd_rows_ex.argtypes = [_dp, _i64, _dp, _i64, _dp, _i64, _dp, _i64,
                                                _dp, _dp, _dp, _int, _int, _int, _dbl, _int,
                                                _int, _ip, _int, _ip, _int]
        lib.oracle_sdpa_fwd_ex.argtypes = [_dp, _dp, _dp, _dp, _dp, _int, _int, _int, _int,
                                           _int, _int, _dbl, _int, _int]
        lib.oracle_sdpa_bwd_ex.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _int, _int, _int,
                                           _int, _int, _int, _dbl, _int, _int]
        lib.oracle_sdpa_varlen_fwd_ex.argtypes = [_dp, _dp, _dp, _dp, _dp, _ip, _ip, _int, _int,
                                                  _int, _int, _dbl, _int, _int]
        lib.oracle_sdpa_varlen_bwd_ex.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _ip, _ip,
                                                  _int, _int, _int, _int, _dbl, _int, _int]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = _dbl
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.POINTER(ctypes.c_uint8), _dp, _i64, _dbl]
        lib.oracle_num_threads.restype = _int
        _lib = lib
        return lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _f64(x) -> np.ndarray:
    """Exact upcast of a (CPU or GPU) tensor / array to a contiguous fp64 array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.int32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _pi(a: np.ndarray):
    return a.ctypes.data_as(_ip)


def sdpa_fwd(q, k, v, scale: float, causal: bool):
    """Dense BHSD forward. q [b,h,s_q,d], k/v [b,h,s_kv,d] -> (o [b,h,s_q,d], lse [b,h,s_q])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s_q, d = q.shape
    s_kv = k.shape[2]
    o = np.zeros((b, h, s_q, d))
    lse = np.zeros((b, h, s_q))
    _load().oracle_sdpa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), b, h, s_q, s_kv, d,
                            float(scale), int(bool(causal)))
    return o, lse


def sdpa_bwd(q, k, v, dout, scale: float, causal: bool):
    """Dense BHSD backward from first principles -> (dq, dk, dv)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    b, h, s_q, d = q.shape
    s_kv = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().oracle_sdpa_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), b, h, s_q,
                            s_kv, d, float(scale), int(bool(causal)))
    return dq, dk, dv


def sdpa_varlen_fwd(q, k, v, cu_q, cu_kv, scale: float, causal: bool):
    """Packed THD forward. q [Tq,h,d], k/v [Tkv,h,d] -> (o [Tq,h,d], lse [Tq,h])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_kv = _i32(cu_q), _i32(cu_kv)
    _, h, d = q.shape
    o = np.zeros_like(q)
    lse = np.full(q.shape[:2], np.nan)
    _load().oracle_sdpa_varlen_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _pi(cu_q), _pi(cu_kv),
                                   len(cu_q) - 1, h, d, float(scale), int(bool(causal)))
    return o, lse


def sdpa_varlen_bwd(q, k, v, dout, cu_q, cu_kv, scale: float, causal: bool):
    """Packed THD backward -> (dq, dk, dv) in the packed layout."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q, cu_kv = _i32(cu_q), _i32(cu_kv)
    _, h, d = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().oracle_sdpa_varlen_bwd(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                                   _pi(cu_q), _pi(cu_kv), len(cu_q) - 1, h, d, float(scale),
                                   int(bool(causal)))
    return dq, dk, dv


def attn_fwd_rows(q, k, v, rows, scale: float, causal: bool):
    """One problem (q [n_q,d], k/v [n_kv,d]); forward of the listed query rows only.

    Returns (o [len(rows), d], lse [len(rows)]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = _i32(rows)
    n_q, d = q.shape
    n_kv = k.shape[0]
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    _load().oracle_attn_fwd_rows(_p(q), d, _p(k), d, _p(v), d, _p(o), _p(lse), n_q, n_kv, d,
                                 float(scale), int(bool(causal)), _pi(rows), len(rows))
    return o, lse


def attn_bwd_rows(q, k, v, dout, q_rows, kv_rows, scale: float, causal: bool):
    """One problem; dQ of the listed query rows and dK/dV of the listed key rows.

    The row statistics are computed for every query row (dK/dV need them).
    Returns (dq [len(q_rows), d], dk [len(kv_rows), d], dv [len(kv_rows), d]).
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    q_rows, kv_rows = _i32(q_rows), _i32(kv_rows)
    n_q, d = q.shape
    n_kv = k.shape[0]
    dq = np.zeros((len(q_rows), d))
    dk = np.zeros((len(kv_rows), d))
    dv = np.zeros((len(kv_rows), d))
    _load().oracle_attn_bwd_rows(_p(q), d, _p(k), d, _p(v), d, _p(dout), d, _p(dq), _p(dk),
                                 _p(dv), n_q, n_kv, d, float(scale), int(bool(causal)),
                                 _pi(q_rows), len(q_rows), _pi(kv_rows), len(kv_rows))
    return dq, dk, dv


# ----------------------------------------------------------------- masks, GQA
#: mask names of the extended entry points: none, causal aligned top-left
#: (query i sees keys j <= i) or bottom-right (j <= i + n_kv - n_q).
MASKS = {"none": 0, "top_left": 1, "bottom_right": 2}


def _mask(mask) -> int:
    return MASKS[mask] if isinstance(mask, str) else int(mask)


def sdpa_fwd_ex(q, k, v, scale: float, mask="top_left", window_left: int = -1):
    """Dense forward with grouped key/value heads and the extended masks.

    q [b,h,s_q,d]; k/v [b,h_kv,s_kv,d] with h a multiple of h_kv (query head
    hq reads key/value head hq // (h // h_kv)).  window_left >= 0 keeps that
    many keys left of the (aligned) diagonal visible.  -> (o, lse).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    o = np.zeros((b, h, s_q, d))
    lse = np.zeros((b, h, s_q))
    _load().oracle_sdpa_fwd_ex(_p(q), _p(k), _p(v), _p(o), _p(lse), b, h, h_kv, s_q, s_kv, d,
                               float(scale), _mask(mask), int(window_left))
    return o, lse


def sdpa_bwd_ex(q, k, v, dout, scale: float, mask="top_left", window_left: int = -1):
    """Dense backward of sdpa_fwd_ex -> (dq [b,h,s_q,d], dk, dv [b,h_kv,s_kv,d])."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    b, h, s_q, d = q.shape
    h_kv, s_kv = k.shape[1], k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().oracle_sdpa_bwd_ex(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv), b, h,
                               h_kv, s_q, s_kv, d, float(scale), _mask(mask), int(window_left))
    return dq, dk, dv


def sdpa_varlen_fwd_ex(q, k, v, cu_q, cu_kv, scale: float, mask="top_left",
                       window_left: int = -1):
    """Packed forward: q [Tq,h,d], k/v [Tkv,h_kv,d] -> (o [Tq,h,d], lse [Tq,h])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    cu_q, cu_kv = _i32(cu_q), _i32(cu_kv)
    _, h, d = q.shape
    h_kv = k.shape[1]
    o = np.zeros_like(q)
    lse = np.full(q.shape[:2], np.nan)
    _load().oracle_sdpa_varlen_fwd_ex(_p(q), _p(k), _p(v), _p(o), _p(lse), _pi(cu_q),
                                      _pi(cu_kv), len(cu_q) - 1, h, h_kv, d, float(scale),
                                      _mask(mask), int(window_left))
    return o, lse


def sdpa_varlen_bwd_ex(q, k, v, dout, cu_q, cu_kv, scale: float, mask="top_left",
                       window_left: int = -1):
    """Packed backward of sdpa_varlen_fwd_ex -> (dq, dk, dv) in the packed layouts."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    cu_q, cu_kv = _i32(cu_q), _i32(cu_kv)
    _, h, d = q.shape
    h_kv = k.shape[1]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _load().oracle_sdpa_varlen_bwd_ex(_p(q), _p(k), _p(v), _p(dout), _p(dq), _p(dk), _p(dv),
                                      _pi(cu_q), _pi(cu_kv), len(cu_q) - 1, h, h_kv, d,
                                      float(scale), _mask(mask), int(window_left))
    return dq, dk, dv


def attn_fwd_rows_ex(q, k, v, rows, scale: float, mask="top_left", window_left: int = -1):
    """One problem (q [n_q,d], k/v [n_kv,d]), listed query rows, extended masks."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    rows = _i32(rows)
    n_q, d = q.shape
    n_kv = k.shape[0]
    o = np.zeros((len(rows), d))
    lse = np.zeros(len(rows))
    _load().oracle_attn_fwd_rows_ex(_p(q), d, _p(k), d, _p(v), d, _p(o), _p(lse), n_q, n_kv, d,
                                    float(scale), _mask(mask), int(window_left), _pi(rows),
                                    len(rows))
    return o, lse


def attn_bwd_rows_ex(q, k, v, dout, q_rows, kv_rows, scale: float, mask="top_left",
                     window_left: int = -1):
    """One problem; dQ of the listed query rows, dK/dV of the listed key rows."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    q_rows, kv_rows = _i32(q_rows), _i32(kv_rows)
    n_q, d = q.shape
    n_kv = k.shape[0]
    dq = np.zeros((len(q_rows), d))
    dk = np.zeros((len(kv_rows), d))
    dv = np.zeros((len(kv_rows), d))
    _load().oracle_attn_bwd_rows_ex(_p(q), d, _p(k), d, _p(v), d, _p(dout), d, _p(dq), _p(dk),
                                    _p(dv), n_q, n_kv, d, float(scale), _mask(mask),
                                    int(window_left), _pi(q_rows), len(q_rows), _pi(kv_rows),
                                    len(kv_rows))
    return dq, dk, dv


# ------------------------------------------------------------------ FP8 inputs
def e4m3_decode(code: int) -> float:
    """Real value of one E4M3 code (see sdpa_oracle.c)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_to_f64(codes, descale: float) -> np.ndarray:
    """Decode an array of E4M3 codes (uint8, any shape) times a per-tensor descale."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            codes = codes.detach().cpu().contiguous().view(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_to_f64(c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), _p(out), c.size,
                               float(descale))
    return out


def sdpa_fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float, scale: float,
                 mask="top_left", window_left: int = -1):
    """Dense forward of E4M3 inputs with per-tensor descales: attention of the
    real values decode(x) * descale_x, in fp64 -> (o, lse)."""
    return sdpa_fwd_ex(e4m3_to_f64(q, descale_q), e4m3_to_f64(k, descale_k),
                       e4m3_to_f64(v, descale_v), scale, mask, window_left)


def sdpa_varlen_fwd_fp8(q, k, v, cu_q, cu_kv, descale_q: float, descale_k: float,
                        descale_v: float, scale: float, mask="top_left", window_left: int = -1):
    """Packed forward of E4M3 inputs with per-tensor descales -> (o, lse)."""
    return sdpa_varlen_fwd_ex(e4m3_to_f64(q, descale_q), e4m3_to_f64(k, descale_k),
                              e4m3_to_f64(v, descale_v), cu_q, cu_kv, scale, mask, window_left)
