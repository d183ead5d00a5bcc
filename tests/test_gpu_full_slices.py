"""Whole-slice parity of the full-size workloads against the fp64 oracle.

Each workload runs on the GPU at its full size, in the launch configuration
the benchmark times; then whole attention slices -- every row and every
column of O, LSE, dQ, dK and dV of a (batch, head) slice, or of one head of
every packed sequence -- are compared element by element with the oracle's
definition of that slice (tolerances: O <= 1e-2 max|ref|, |dLSE| <= 1e-3,
dQ/dK/dV <= 2e-2 max|ref|, per slice; packed results also per sequence, as
cudnn-frontend PR #554 checks THD results against per-sequence references).

Slices checked:
- b1 h32 s16384 d128 causal (Q, K doubled): heads 0, 3, 4 and 31.  The
  backward runs its CTAs in groups of four key/value slices, so heads 3 and 4
  sit on both sides of the first group boundary, 0 and 31 at the ends of the
  order.  The forward runs on both forward kernels.
- 16 packed sequences, h32 d128 causal: heads 0 and 31 of every sequence.
- b2 h16 s4096 d128 non-causal: (0, 0), (0, 3), (0, 4) and (1, 15), the same
  group boundary and both ends.
"""
import pytest
import torch

import oracle_refs
import sdpa_inputs
from helpers import GRAD_TOL, O_TOL, check_lse, check_rel

pytestmark = pytest.mark.gpu

C3 = "c3_b2h16s4096d128_noncausal"
C4 = "c4_thd16_h32d128_causal"
C5 = "c5_b1h32s16384d128_causal_qk2"
C5_SLICES = ((0, 0), (0, 3), (0, 4), (0, 31))
C3_SLICES = ((0, 0), (0, 3), (0, 4), (1, 15))
C4_HEADS = (0, 31)
DENSE_SLICES = {C3: C3_SLICES, C5: C5_SLICES}
OTOL = O_TOL[torch.bfloat16]


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def _finite(*xs):
    for x in xs:
        assert torch.isfinite(x.float()).all()


def _dense_run(sdpa, name, variant=0, backward=False):
    """The workload's forward (on the given forward kernel choice) and, if
    asked, its backward; CPU copies of the outputs."""
    w = sdpa_inputs.WORKLOADS[name]
    t = oracle_refs.inputs(name)
    q, k, v = (t[x].cuda() for x in ("q", "k", "v"))
    sdpa.sdpa_set_forward_variant(variant)
    try:
        o, lse = sdpa.attention(q, k, v, scale=w.scale, causal=w.causal)
    finally:
        sdpa.sdpa_set_forward_variant(0)
    grads = ()
    if backward:
        grads = sdpa.attention_bwd(q, k, v, o, t["do"].cuda(), lse, scale=w.scale,
                                   causal=w.causal)
    torch.cuda.synchronize()
    sdpa.sdpa_check_device_error()
    return tuple(x.cpu() for x in (o, lse) + tuple(grads))


def _packed_run(sdpa, variant=0, backward=False):
    w = sdpa_inputs.WORKLOADS[C4]
    t = oracle_refs.inputs(C4)
    lens = t["lengths"]
    q, k, v = (t[x].cuda() for x in ("q", "k", "v"))
    cu_q, cu_kv = t["cu_q"].cuda(), t["cu_kv"].cuda()
    sdpa.sdpa_set_forward_variant(variant)
    try:
        o, lse = sdpa.attention_varlen(q, k, v, cu_q, cu_kv, max(lens), max(lens),
                                       scale=w.scale, causal=w.causal)
    finally:
        sdpa.sdpa_set_forward_variant(0)
    grads = ()
    if backward:
        grads = sdpa.attention_varlen_bwd(q, k, v, o, t["do"].cuda(), lse, cu_q, cu_kv,
                                          max(lens), max(lens), scale=w.scale, causal=w.causal)
    torch.cuda.synchronize()
    sdpa.sdpa_check_device_error()
    return tuple(x.cpu() for x in (o, lse) + tuple(grads))


@pytest.mark.parametrize("variant", [1, 2], ids=["one_tile", "two_tile"])
@pytest.mark.parametrize("name", [C3, C5])
def test_full_size_dense_fwd_whole_slices(sdpa, name, variant):
    o, lse = _dense_run(sdpa, name, variant)
    _finite(o, lse)
    for bb, hh in DENSE_SLICES[name]:
        r_o, r_lse = oracle_refs.dense_slice(name, bb, hh, True)[:2]
        check_rel(o[bb, hh], r_o, OTOL, f"O[{bb},{hh}]")
        check_lse(lse[bb, hh], r_lse, f"lse[{bb},{hh}]")


@pytest.mark.usefixtures("bwd_kernel")
@pytest.mark.parametrize("name", [C3, C5])
def test_full_size_dense_bwd_whole_slices(sdpa, name):
    o, lse, dq, dk, dv = _dense_run(sdpa, name, 0, backward=True)
    _finite(o, lse, dq, dk, dv)
    for bb, hh in DENSE_SLICES[name]:
        r = oracle_refs.dense_slice(name, bb, hh, True)
        check_rel(o[bb, hh], r[0], OTOL, f"O[{bb},{hh}]")
        check_lse(lse[bb, hh], r[1], f"lse[{bb},{hh}]")
        for g, rr, nm in zip((dq, dk, dv), r[2:], ("dq", "dk", "dv")):
            check_rel(g[bb, hh], rr, GRAD_TOL, f"{nm}[{bb},{hh}]")


def _per_sequence(cu, got, ref, tol, name):
    for n in range(len(cu) - 1):
        a, e = cu[n], cu[n + 1]
        if e > a:
            check_rel(got[a:e], ref[a:e], tol, f"{name} seq {n}")


@pytest.mark.parametrize("variant", [1, 2], ids=["one_tile", "two_tile"])
def test_full_size_packed_fwd_every_sequence(sdpa, variant):
    o, lse = _packed_run(sdpa, variant)
    _finite(o, lse)
    cu = oracle_refs.inputs(C4)["cu_q"].tolist()
    for hh in C4_HEADS:
        r_o, r_lse = oracle_refs.packed_head(C4, hh, True)[:2]
        _per_sequence(cu, o[:, hh], r_o, OTOL, f"O head {hh}")
        check_lse(lse[:, hh], r_lse, f"lse head {hh}")


@pytest.mark.usefixtures("bwd_kernel")
def test_full_size_packed_bwd_every_sequence(sdpa):
    o, lse, dq, dk, dv = _packed_run(sdpa, 0, backward=True)
    _finite(o, lse, dq, dk, dv)
    cu = oracle_refs.inputs(C4)["cu_q"].tolist()
    for hh in C4_HEADS:
        r = oracle_refs.packed_head(C4, hh, True)
        _per_sequence(cu, o[:, hh], r[0], OTOL, f"O head {hh}")
        check_lse(lse[:, hh], r[1], f"lse head {hh}")
        for g, rr, nm in zip((dq, dk, dv), r[2:], ("dq", "dk", "dv")):
            _per_sequence(cu, g[:, hh], rr, GRAD_TOL, f"{nm} head {hh}")
            check_rel(g[:, hh], rr, GRAD_TOL, f"{nm} head {hh} (whole)")

