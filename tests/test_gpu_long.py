"""Parity on sequences four times longer than the long-context workload's.

Key/value slices of 65,536 tokens, bf16 N(0, 1) inputs from sdpa_inputs.dense,
scale 1/sqrt(d):
- causal (top-left), one head, at d = 128 and d = 64: the forward's units walk up
  to 512 key tiles and the backward's units up to 512 query tiles, four times the
  16,384-token workload's (d = 64 runs the other TMEM layout: dQ has columns of
  its own and dO two stages);
- the FP8 (E4M3) forward of the d = 128 causal head, within the bound derived for
  E4M3 P;
- a packed list of one 40,997-token sequence among short and ragged ones (1 to 2049
  tokens), two query heads on one key/value head, causal (sequences shorter than 8
  tokens have their gradients checked by the whole-tensor tests only, reading 8);
- a bottom-right band (window_left 5000) with s_q = 61,000 (a ragged last
  query tile) against s_kv = 65,536, two query heads on one key/value head,
  d = 128.

Rows are sampled and the oracle computes them one by one (attn_fwd_rows /
attn_bwd_rows and their masked forms).  Key rows need every query row's
statistics, about 1.1 TFLOP of fp64 work for the causal head, so the
references are computed once per process.  Both backward main kernels run
each case.

Tolerances are those of helpers.py, relative to a tensor's largest reference
value.  On a sample that maximum can only be underestimated, and under a
causal mask the largest dQ, O, dK and dV values sit in the first rows, which
see few keys.  So the sample holds the first two query and key tiles whole,
besides the tile boundaries, the middle, the last rows and seeded random rows.
Those first rows are also where the backward's inherent error is largest: D =
rowsum(dO * O) is formed from the 16-bit O the backward is given, and a row
that sees two keys has a dQ that is a difference of nearly equal terms (row 1
of the causal case: about 3 % of that row, which an emulation of the same
rounding on the CPU reproduces).
"""
import functools
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import GRAD_TOL, O_TOL, check_lse, check_rel

pytestmark = pytest.mark.gpu

CASES = {
    "causal_s65536": dict(d=128, h=1, h_kv=1, s_q=65536, s_kv=65536, mask="top_left", window=-1,
                          seed=65536),
    "causal_s65536_d64": dict(d=64, h=1, h_kv=1, s_q=65536, s_kv=65536, mask="top_left",
                              window=-1, seed=65537),
    "band_gqa_s61000_s65536": dict(d=128, h=2, h_kv=1, s_q=61000, s_kv=65536, mask="bottom_right",
                                   window=5000, seed=61000),
}


def _scale(c):
    return 1.0 / math.sqrt(c["d"])


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def _rows(n, seed):
    g = np.random.default_rng(seed)
    base = set(range(min(n, 256)))
    base |= {n // 2 - 1, n // 2, n - 129, n - 128, n - 2, n - 1}
    base |= set(g.integers(0, n, 8).tolist())
    return np.array(sorted(r for r in base if 0 <= r < n), np.int32)


@functools.lru_cache(maxsize=None)
def _inputs(name):
    c = CASES[name]
    return sdpa_inputs.dense(1, c["h"], c["s_q"], c["s_kv"], c["d"], seed=c["seed"],
                             h_kv=c["h_kv"])


@functools.lru_cache(maxsize=None)
def _reference(name):
    """Sampled rows of every query head: (q_rows, kv_rows, o, lse, dq) per
    head, and dK/dV rows per key/value head (summed over its query heads)."""
    c = CASES[name]
    q, k, v, do = _inputs(name)
    group = c["h"] // c["h_kv"]
    q_rows, kv_rows = _rows(c["s_q"], c["seed"] + 1), _rows(c["s_kv"], c["seed"] + 2)
    o, lse, dq = [], [], []
    dk = [np.zeros((len(kv_rows), c["d"])) for _ in range(c["h_kv"])]
    dv = [np.zeros((len(kv_rows), c["d"])) for _ in range(c["h_kv"])]
    for hq in range(c["h"]):
        hk = hq // group
        args = (q[0, hq], k[0, hk], v[0, hk])
        ro, rl = oracle.attn_fwd_rows_ex(*args, q_rows, _scale(c), c["mask"], c["window"])
        rdq, rdk, rdv = oracle.attn_bwd_rows_ex(*args, do[0, hq], q_rows, kv_rows, _scale(c),
                                                c["mask"], c["window"])
        o.append(ro)
        lse.append(rl)
        dq.append(rdq)
        dk[hk] += rdk
        dv[hk] += rdv
    return q_rows, kv_rows, o, lse, dq, dk, dv


@pytest.mark.usefixtures("bwd_kernel")
@pytest.mark.parametrize("name", list(CASES))
def test_long_sequence_sampled_rows(sdpa, name):
    c = CASES[name]
    q, k, v, do = (x.cuda() for x in _inputs(name))
    o, lse = sdpa.attention(q, k, v, scale=_scale(c), mask=c["mask"], window_left=c["window"])
    dq, dk, dv = sdpa.attention_bwd(q, k, v, o, do, lse, scale=_scale(c), mask=c["mask"],
                                    window_left=c["window"])
    torch.cuda.synchronize()
    q_rows, kv_rows, ro, rl, rdq, rdk, rdv = _reference(name)
    qi, ki = torch.from_numpy(q_rows).long(), torch.from_numpy(kv_rows).long()
    o, lse, dq, dk, dv = (x.cpu() for x in (o, lse, dq, dk, dv))
    for hq in range(c["h"]):
        check_rel(o[0, hq, qi], ro[hq], O_TOL[torch.bfloat16], f"o[{hq}]")
        check_lse(lse[0, hq, qi], rl[hq], f"lse[{hq}]")
        check_rel(dq[0, hq, qi], rdq[hq], GRAD_TOL, f"dq[{hq}]")
    for hk in range(c["h_kv"]):
        check_rel(dk[0, hk, ki], rdk[hk], GRAD_TOL, f"dk[{hk}]")
        check_rel(dv[0, hk, ki], rdv[hk], GRAD_TOL, f"dv[{hk}]")


@functools.lru_cache(maxsize=None)
def _fp8_reference(name):
    """The E4M3 encoding of the case's inputs (codes, descales), the decoded
    values and the oracle's rows of the forward on them (query head 0)."""
    c = CASES[name]
    q, k, v, _ = _inputs(name)
    enc = [sdpa_inputs.fp8_quantize(x.float()) for x in (q, k, v)]
    (qc, dsq), (kc, dsk), (vc, dsv) = enc
    qd = oracle.e4m3_to_f64(qc[0, 0], dsq)
    kd = oracle.e4m3_to_f64(kc[0, 0], dsk)
    vd = oracle.e4m3_to_f64(vc[0, 0], dsv)
    q_rows = _rows(c["s_q"], c["seed"] + 3)
    ro, rl = oracle.attn_fwd_rows_ex(qd, kd, vd, q_rows, _scale(c), c["mask"], c["window"])
    return enc, q_rows, ro, rl, float(np.abs(vd).max())


def test_long_sequence_fp8_forward_sampled_rows(sdpa):
    """The FP8 forward over the 65,536-token causal head: O within the bound
    derived for E4M3 P (2^-4 max|V| + 2^-8 max|O| of the oracle on the decoded
    inputs), LSE within 1e-3."""
    name = "causal_s65536"
    c = CASES[name]
    enc, q_rows, ro, rl, vmax = _fp8_reference(name)
    (qc, dsq), (kc, dsk), (vc, dsv) = enc
    ds = [torch.tensor([x], dtype=torch.float32, device="cuda") for x in (dsq, dsk, dsv)]
    o, lse, _ = sdpa.attention_fp8(qc.cuda(), kc.cuda(), vc.cuda(), *ds, scale=_scale(c),
                                   causal=True)
    torch.cuda.synchronize()
    qi = torch.from_numpy(q_rows).long()
    o, lse = o[0, 0, qi].cpu(), lse[0, 0, qi].cpu()
    assert torch.isfinite(o.float()).all()
    err = float(np.abs(o.double().numpy() - ro).max())
    bound = 2.0 ** -4 * vmax + 2.0 ** -8 * float(np.abs(ro).max()) + 1e-6
    assert err <= bound, f"max|dO| {err:.3e} > bound {bound:.3e}"
    check_lse(lse, rl, "lse")


# A packed list with one long sequence among short and ragged ones, two query
# heads on one key/value head, causal: the packed forward takes the long
# sequence's units first and the short ones on demand; the backward walks up
# to 321 query tiles per unit.
PACKED_LENS = [40997, 1, 127, 128, 129, 700, 2049, 33]


@functools.lru_cache(maxsize=None)
def _packed_inputs():
    return sdpa_inputs.packed(PACKED_LENS, PACKED_LENS, 2, 128, seed=40997, h_kv=1)


@functools.lru_cache(maxsize=None)
def _packed_reference():
    """Per sequence: its sampled rows, O/LSE/dQ rows per query head and dK/dV
    rows summed over the two query heads."""
    q, k, v, do, cu, _ = _packed_inputs()
    scale = 1.0 / math.sqrt(128)
    out = []
    for n, L in enumerate(PACKED_LENS):
        t0 = int(cu[n])
        rows = np.arange(L, dtype=np.int32) if L <= 300 else _rows(L, 7 + n)
        o, lse, dq = [], [], []
        dk = np.zeros((len(rows), 128))
        dv = np.zeros((len(rows), 128))
        for hq in range(2):
            args = (q[t0:t0 + L, hq], k[t0:t0 + L, 0], v[t0:t0 + L, 0])
            ro, rl = oracle.attn_fwd_rows_ex(*args, rows, scale, "top_left", -1)
            rdq, rdk, rdv = oracle.attn_bwd_rows_ex(*args, do[t0:t0 + L, hq], rows, rows, scale,
                                                    "top_left", -1)
            o.append(ro)
            lse.append(rl)
            dq.append(rdq)
            dk += rdk
            dv += rdv
        out.append((t0, rows, o, lse, dq, dk, dv))
    return out


@pytest.mark.usefixtures("bwd_kernel")
def test_long_packed_sequence_sampled_rows(sdpa):
    q, k, v, do, cu, _ = (x.cuda() for x in _packed_inputs())
    mx = max(PACKED_LENS)
    scale = 1.0 / math.sqrt(128)
    o, lse = sdpa.attention_varlen(q, k, v, cu, cu, mx, mx, scale=scale, causal=True)
    dq, dk, dv = sdpa.attention_varlen_bwd(q, k, v, o, do, lse, cu, cu, mx, mx, scale=scale,
                                           causal=True)
    torch.cuda.synchronize()
    o, lse, dq, dk, dv = (x.cpu() for x in (o, lse, dq, dk, dv))
    for n, (t0, rows, ro, rl, rdq, rdk, rdv) in enumerate(_packed_reference()):
        idx = torch.from_numpy(rows).long() + t0
        for hq in range(2):
            check_rel(o[idx, hq], ro[hq], O_TOL[torch.bfloat16], f"o[seq {n}, head {hq}]")
            check_lse(lse[idx, hq], rl[hq], f"lse[seq {n}, head {hq}]")
            if PACKED_LENS[n] >= 8:
                check_rel(dq[idx, hq], rdq[hq], GRAD_TOL, f"dq[seq {n}, head {hq}]")
        if PACKED_LENS[n] >= 8:
            check_rel(dk[idx, 0], rdk, GRAD_TOL, f"dk[seq {n}]")
            check_rel(dv[idx, 0], rdv, GRAD_TOL, f"dv[seq {n}]")
