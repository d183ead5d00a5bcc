"""Cached fp64 oracle references of whole attention slices of the configured
workloads (test infrastructure).

One (batch, head) slice of a dense problem, or one head of a packed problem,
is an independent attention problem, so its reference is the oracle's dense or
packed entry point applied to that slice alone.  The references are computed
once per pytest process and shared by every test file that checks the same
slice (the plain, deterministic and variant backward runs of one workload).
"""
from __future__ import annotations

import functools

import oracle
import sdpa_inputs


@functools.lru_cache(maxsize=None)
def inputs(name: str):
    """All CPU input tensors of a named workload (drawn once)."""
    return sdpa_inputs.make(sdpa_inputs.WORKLOADS[name])


@functools.lru_cache(maxsize=None)
def dense_slice(name: str, bb: int, hh: int, backward: bool):
    """(o, lse) of slice (bb, hh), plus (dq, dk, dv) when backward; each
    without the leading (1, 1) batch and head axes."""
    w = sdpa_inputs.WORKLOADS[name]
    t = inputs(name)
    sl = [t[x][bb:bb + 1, hh:hh + 1] for x in ("q", "k", "v", "do")]
    o, lse = oracle.sdpa_fwd(sl[0], sl[1], sl[2], w.scale, w.causal)
    out = [o[0, 0], lse[0, 0]]
    if backward:
        dq, dk, dv = oracle.sdpa_bwd(*sl, w.scale, w.causal)
        out += [dq[0, 0], dk[0, 0], dv[0, 0]]
    return tuple(out)


@functools.lru_cache(maxsize=None)
def packed_head(name: str, hh: int, backward: bool):
    """(o [T, d], lse [T]) of head hh over every packed sequence, plus
    (dq, dk, dv) when backward."""
    w = sdpa_inputs.WORKLOADS[name]
    t = inputs(name)
    sl = [t[x][:, hh:hh + 1] for x in ("q", "k", "v", "do")]
    o, lse = oracle.sdpa_varlen_fwd(sl[0], sl[1], sl[2], t["cu_q"], t["cu_kv"], w.scale,
                                    w.causal)
    out = [o[:, 0], lse[:, 0]]
    if backward:
        dq, dk, dv = oracle.sdpa_varlen_bwd(*sl, t["cu_q"], t["cu_kv"], w.scale, w.causal)
        out += [dq[:, 0], dk[:, 0], dv[:, 0]]
    return tuple(out)
