"""The forwards taking their units dynamically: packed lists run sequence by
sequence (longest first, from each CTA's table of the sequences) -- on the
one-tile kernel when their K and V outgrow 64 MiB, on the two-tile kernel
always -- and those launches take their units from a counter instead of a
fixed deal of the list.  Every case runs on both kernels; every sequence is
checked against the fp64 oracle.

Tolerances: O within 1e-2 of max|O_ref| per sequence (16-bit), LSE within
1e-3; FP8 within the derived bound of tests/test_gpu_fp8.py (2^-4 max|V| +
2^-8 max|O_ref|).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import O_TOL, check_lse, check_rel, np64

pytestmark = pytest.mark.gpu

SLICE_MAJOR_KV_BYTES = 64 << 20  # above this K + V, packed lists go sequence by sequence


@pytest.fixture(scope="module", params=[1, 2], ids=["one_tile", "two_tile"])
def sdpa(request):
    import scaled_dot_product_04_gb300 as m
    m.load()
    m.sdpa_set_forward_variant(request.param)
    yield m
    m.sdpa_set_forward_variant(0)


def _lengths(n, lo, hi, seed, zero_q=(), zero_kv=()):
    g = np.random.default_rng(seed)
    lq = g.integers(lo, hi + 1, n).tolist()
    lk = list(lq)
    for i in zero_q:
        lq[i] = 0
    for i in zero_kv:
        lk[i] = 0
    return lq, lk


def _per_sequence(cu, got, ref, tol, name):
    for n in range(len(cu) - 1):
        a, e = cu[n], cu[n + 1]
        if e > a:
            check_rel(got[a:e], ref[a:e], tol, f"{name} seq {n}")


@pytest.mark.parametrize("d,n,lo,hi,h,mask", [
    (128, 12, 64, 3000, 16, "top_left"),
    (128, 14, 64, 3000, 16, "bottom_right"),   # with a sequence without queries and one without keys
    (64, 60, 100, 1200, 32, "top_left"),
])
def test_dynamic_packed_every_sequence(sdpa, d, n, lo, hi, h, mask):
    zq, zk = ((3,), (7,)) if mask == "bottom_right" else ((), ())
    lq, lk = _lengths(n, lo, hi, seed=n + d, zero_q=zq, zero_kv=zk)
    assert 2 * sum(lk) * h * d * 2 > SLICE_MAJOR_KV_BYTES
    q, k, v, _, cu_q, cu_kv = sdpa_inputs.packed(lq, lk, h, d, seed=n)
    scale = 1.0 / math.sqrt(d)
    o, lse = sdpa.attention_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_kv.cuda(), max(lq),
                                   max(lk), scale=scale, mask=mask)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_varlen_fwd_ex(q, k, v, cu_q, cu_kv, scale, mask, -1)
    cu = cu_q.tolist()
    _per_sequence(cu, o, ro, O_TOL[torch.bfloat16], "o")
    check_lse(lse, rlse)


def test_dynamic_packed_fp8(sdpa):
    lq, lk = _lengths(12, 64, 3000, seed=5)
    h, d = 32, 128
    assert 2 * sum(lk) * h * d > SLICE_MAJOR_KV_BYTES
    qc, kc, vc, dq, dk, dv, cu_q, cu_kv = sdpa_inputs.fp8_packed(lq, lk, h, d, seed=95)
    scale = 1.0 / math.sqrt(d)
    T = qc.shape[0]
    sc = lambda x: torch.tensor([x], dtype=torch.float32, device="cuda")  # noqa: E731
    o = torch.empty(T, h, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, h, dtype=torch.float32, device="cuda")
    sdpa.sdpa_varlen_fwd_fp8(qc.cuda(), kc.cuda(), vc.cuda(), o, lse, sc(dq), sc(dk), sc(dv), None,
                             None, cu_q.cuda(), cu_kv.cuda(), len(lq), T, kc.shape[0], max(lq),
                             max(lk), h, h, d, scale, 1, -1, 0)
    torch.cuda.synchronize()
    ro, rlse = oracle.sdpa_varlen_fwd_fp8(qc, kc, vc, cu_q, cu_kv, dq, dk, dv, scale, "top_left")
    vmax = float(np.abs(oracle.e4m3_to_f64(vc, dv)).max())
    err = float(np.abs(np64(o) - ro).max())
    bound = 2.0 ** -4 * vmax + 2.0 ** -8 * float(np.abs(ro).max()) + 1e-6
    assert err <= bound, f"max|dO| {err:.3e} > bound {bound:.3e}"
    check_lse(lse, rlse)


def test_dynamic_packed_repeatable(sdpa):
    """The units run in whatever order the CTAs take them; each unit's
    arithmetic is fixed, so two runs give the same bits."""
    lq, lk = _lengths(12, 64, 3000, seed=12 + 128)
    h, d = 16, 128
    q, k, v, _, cu_q, cu_kv = (x.cuda() for x in sdpa_inputs.packed(lq, lk, h, d, seed=12))
    a = sdpa.attention_varlen(q, k, v, cu_q, cu_kv, max(lq), max(lk), scale=0.088, causal=True)
    b = sdpa.attention_varlen(q, k, v, cu_q, cu_kv, max(lq), max(lk), scale=0.088, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
