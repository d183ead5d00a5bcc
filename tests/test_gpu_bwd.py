"""Backward parity: CUDA dQ/dK/dV (through the C ABI, fed by the CUDA
forward's O and LSE) vs the fp64 oracle's analytic gradients.

Tolerance: max|got - ref| <= 2e-2 * max|ref| per tensor (and per sequence for
packed inputs).  The full-size workloads are compared whole slice by whole
slice in test_gpu_full_slices.py.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import GRAD_TOL, check_rel, np64

# every test here runs on each backward main kernel (tests/conftest.py)
pytestmark = [pytest.mark.gpu, pytest.mark.usefixtures("bwd_variant")]


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    return m


def _dense_bwd(sdpa, q, k, v, do, scale, causal):
    q, k, v, do = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = sdpa.attention_bwd(q, k, v, o, do, lse, scale=scale, causal=causal)
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s_q,s_kv", [(333, 333), (1, 1), (256, 256), (200, 461), (461, 200)])
def test_dense_bwd_shapes(sdpa, d, causal, s_q, s_kv):
    q, k, v, do = sdpa_inputs.dense(2, 3, s_q, s_kv, d, seed=s_q + 3 * s_kv)
    scale = 1.0 / math.sqrt(d)
    got = _dense_bwd(sdpa, q, k, v, do, scale, causal)
    ref = oracle.sdpa_bwd(q, k, v, do, scale, causal)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        if np.abs(r).max() == 0:
            # e.g. one visible key: dQ is exactly 0, but D comes from the
            # rounded O, so only rounding noise may remain
            assert float(g.abs().max()) <= 1e-4, name
        else:
            check_rel(g, r, GRAD_TOL, name)


@pytest.mark.parametrize("d", [64, 128])
def test_dense_bwd_fp16(sdpa, d):
    q, k, v, do = sdpa_inputs.dense(1, 4, 300, 300, d, seed=99, dtype=torch.float16)
    scale = 1.0 / math.sqrt(d)
    got = _dense_bwd(sdpa, q, k, v, do, scale, True)
    ref = oracle.sdpa_bwd(q, k, v, do, scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_rel(g, r, GRAD_TOL, name)


def test_dense_bwd_sharpened(sdpa):
    q, k, v, do = sdpa_inputs.dense(1, 2, 1000, 1000, 128, seed=1005, qk_mult=2.0)
    scale = 1.0 / math.sqrt(128)
    got = _dense_bwd(sdpa, q, k, v, do, scale, True)
    ref = oracle.sdpa_bwd(q, k, v, do, scale, True)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        check_rel(g, r, GRAD_TOL, name)


def test_dkdv_deterministic(sdpa):
    q, k, v, do = (x.cuda() for x in sdpa_inputs.dense(1, 4, 700, 700, 128, seed=5))
    o, lse = sdpa.attention(q, k, v, scale=0.088, causal=True)
    a = sdpa.attention_bwd(q, k, v, o, do, lse, scale=0.088, causal=True)
    b = sdpa.attention_bwd(q, k, v, o, do, lse, scale=0.088, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    check_rel(a[0], b[0].double().cpu().numpy(), 1e-2, "dq rerun")


def test_bwd_no_queries(sdpa):
    k = torch.randn(1, 2, 100, 64, device="cuda").bfloat16()
    q = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 0, device="cuda")
    dq, dk, dv = sdpa.attention_bwd(q, k, k, q, q, lse, scale=0.125, causal=False)
    torch.cuda.synchronize()
    assert torch.all(dk == 0) and torch.all(dv == 0)


def test_bwd_workspace_checks(sdpa):
    q, k, v, do = (x.cuda() for x in sdpa_inputs.dense(1, 2, 128, 128, 64, seed=6))
    o, lse = sdpa.attention(q, k, v, scale=0.125, causal=True)
    need = sdpa.sdpa_bwd_workspace_size(1, 2, 128, 64)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    with pytest.raises(sdpa.SdpaError) as e:
        sdpa.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, 1, 2, 128, 128, 64, 0.125, 1, 0, small,
                      small.numel())
    assert e.value.status == 4


def test_bwd_no_host_sync(sdpa):
    q, k, v, do = (x.cuda() for x in sdpa_inputs.dense(1, 2, 256, 256, 128, seed=7))
    o, lse = sdpa.attention(q, k, v, scale=0.088, causal=True)
    ws = torch.empty(sdpa.sdpa_bwd_workspace_size(1, 2, 256, 128), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        sdpa.sdpa_bwd(q, k, v, o, do, lse, dq, dk, dv, 1, 2, 256, 256, 128, 0.088, 1, 0, ws,
                      ws.numel())
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()


# ------------------------------------------------------------------ packed
PER_SEQ_MIN = 8


def _varlen_bwd_case(sdpa, lens_q, lens_kv, h, d, causal, dtype=torch.bfloat16, seed=0, pad=0):
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lens_q, lens_kv, h, d, seed=seed, dtype=dtype)
    tq, tkv = q.shape[0], k.shape[0]
    scale = 1.0 / math.sqrt(d)

    def g(x):
        if pad == 0:
            return x.cuda()
        buf = torch.full((x.shape[0] + pad,) + tuple(x.shape[1:]), float("nan"), dtype=x.dtype,
                         device="cuda")
        buf[:x.shape[0]] = x.cuda()
        return buf

    qg, kg, vg, dog = g(q), g(k), g(v), g(do)
    cq, ck = cu_q.cuda(), cu_kv.cuda()
    mq, mk = max(lens_q), max(lens_kv)
    o, lse = sdpa.attention_varlen(qg, kg, vg, cq, ck, mq, mk, scale=scale, causal=causal,
                                   total_q=tq, total_kv=tkv)
    dq, dk, dv = sdpa.attention_varlen_bwd(qg, kg, vg, o, dog, lse, cq, ck, mq, mk, scale=scale,
                                           causal=causal, total_q=tq, total_kv=tkv)
    torch.cuda.synchronize()
    dq, dk, dv = dq[:tq], dk[:tkv], dv[:tkv]
    ref = oracle.sdpa_varlen_bwd(q, k, v, do, cu_q, cu_kv, scale, causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        check_rel(got, r, GRAD_TOL, name)
    # Per sequence as well, for sequences of at least PER_SEQ_MIN query rows and
    # keys: with fewer, a gradient can be one small difference dP - D, where D
    # comes from the bf16 output O, and its own relative error reach a few
    # percent (the whole-tensor check above still covers those sequences).
    cq_l, ck_l = cu_q.tolist(), cu_kv.tolist()
    for n in range(len(lens_q)):
        big = min(lens_q[n], lens_kv[n]) >= PER_SEQ_MIN
        for name, got, r, cu in zip(("dq", "dk", "dv"), (dq, dk, dv), ref, (cq_l, ck_l, ck_l)):
            a, e = cu[n], cu[n + 1]
            if e > a and np.abs(r[a:e]).max() > 0:
                if big:
                    check_rel(got[a:e], r[a:e], GRAD_TOL, f"{name} seq {n}")
            elif e > a:
                assert float(got[a:e].abs().max()) <= 1e-4, f"{name} seq {n} should be 0"


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bwd_mixed(sdpa, d, causal):
    lens = [1, 127, 128, 129, 397, 0, 513, 64]
    _varlen_bwd_case(sdpa, lens, lens, 3, d, causal, seed=21)


@pytest.mark.parametrize("n_seqs,lo,hi", [(20, 0, 400), (40, 1, 300), (300, 0, 64), (1100, 0, 24)])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bwd_many_sequences(sdpa, n_seqs, lo, hi, causal):
    """The backward's grid over many packed sequences: each CTA finds its key
    tile in a table of the sequences, built in registers up to 32 sequences,
    in shared memory sorted longest first up to 256 and in list order up to
    1024; longer lists use the envelope grid.  Query and key lengths differ
    per sequence (some zero), so some rows and some key tiles see nothing."""
    g = np.random.default_rng(n_seqs)
    lens_q = g.integers(lo, hi + 1, n_seqs).tolist()
    lens_kv = g.integers(lo, hi + 1, n_seqs).tolist()
    for n in range(0, n_seqs, 97):  # zero-length sequences on either side
        lens_q[n] = 0
        lens_kv[(n + 48) % n_seqs] = 0
    _varlen_bwd_case(sdpa, lens_q, lens_kv, 2, 64, causal, seed=60 + n_seqs)


@pytest.mark.parametrize("n_seqs", [40, 300])
def test_varlen_bwd_many_sequences_gqa_window(sdpa, n_seqs):
    """The same tables with grouped key/value heads (dK, dV summed over each
    group inside one CTA) and a bottom-right band."""
    g = np.random.default_rng(7 * n_seqs)
    lens_q = g.integers(1, 200, n_seqs).tolist()
    lens_kv = g.integers(1, 260, n_seqs).tolist()
    h, h_kv, d = 4, 2, 128
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lens_q, lens_kv, h, d, seed=n_seqs, h_kv=h_kv)
    qg, kg, vg, dog, cq, ck = (x.cuda() for x in (q, k, v, do, cu_q, cu_kv))
    mq, mk = max(lens_q), max(lens_kv)
    o, lse = sdpa.attention_varlen(qg, kg, vg, cq, ck, mq, mk, scale=0.09, mask="bottom_right",
                                   window_left=70)
    got = sdpa.attention_varlen_bwd(qg, kg, vg, o, dog, lse, cq, ck, mq, mk, scale=0.09,
                                    mask="bottom_right", window_left=70)
    torch.cuda.synchronize()
    ref = oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_kv, 0.09, "bottom_right", 70)
    for name, x, r in zip(("dq", "dk", "dv"), got, ref):
        check_rel(x, r, GRAD_TOL, name)


def test_varlen_bwd_nan_capacity_tail(sdpa):
    lens = [100, 200, 97]
    _varlen_bwd_case(sdpa, lens, lens, 4, 128, True, seed=22, pad=300)


def test_varlen_bwd_zero_length_kv(sdpa):
    _varlen_bwd_case(sdpa, [50, 70, 130], [50, 0, 200], 2, 128, False, seed=23)
    _varlen_bwd_case(sdpa, [50, 0, 130], [50, 90, 200], 2, 64, True, seed=24)


def test_varlen_bwd_fp16(sdpa):
    _varlen_bwd_case(sdpa, [300, 17, 256], [300, 17, 256], 2, 128, True, dtype=torch.float16,
                     seed=25)


def test_device_error_word_clean_after_bwd(sdpa):
    sdpa.sdpa_check_device_error()
