"""The backward's two main kernels: which one the automatic choice takes, and
the persistent kernel on lists of many units per CTA (the dynamic unit
counter, the unit ring wrapping around, units that no query sees mixed with
live ones) against the fp64 oracle and against the one-CTA-per-unit kernel.

Tolerance: max|got - ref| <= 2e-2 * max|ref| per tensor; dK and dV of the two
kernels agree bit for bit (the same products in the same order per unit), dQ
to rounding (its fp32 additions may arrive in another order).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from helpers import GRAD_TOL, check_rel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdpa():
    import scaled_dot_product_04_gb300 as m
    m.load()
    yield m
    m.sdpa_set_backward_variant(0)
    m.sdpa_set_backward_grid_limit(0)


def _dense(sdpa, b, h, h_kv, s_q, s_kv, d, mask, window, seed, deterministic=False):
    q, k, v, do = sdpa_inputs.dense(b, h, s_q, s_kv, d, seed=seed, h_kv=h_kv)
    scale = 1.0 / math.sqrt(d)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = sdpa.attention(qc, kc, vc, scale=scale, mask=mask, window_left=window)

    def run():
        g = sdpa.attention_bwd(qc, kc, vc, o, doc, lse, scale=scale, mask=mask, window_left=window,
                               deterministic=deterministic)
        torch.cuda.synchronize()
        return g, sdpa.sdpa_last_backward_variant()
    return (q, k, v, do, scale), run


def _set(sdpa, variant, limit=0):
    sdpa.sdpa_set_backward_variant(variant)
    sdpa.sdpa_set_backward_grid_limit(limit)


def test_automatic_choice(sdpa):
    _set(sdpa, 0)
    # short units (a causal 1024-row problem at d = 64): persistent
    _, run = _dense(sdpa, 1, 2, 2, 1024, 1024, 64, "top_left", -1, 1)
    assert run()[1] == 2
    # long units (32 query tiles per key tile, no mask): one CTA per unit
    _, run = _dense(sdpa, 1, 1, 1, 4096, 4096, 128, "none", -1, 2)
    assert run()[1] == 1
    # a mean of 8.5 query tiles per unit (causal, 16 key tiles): one CTA per unit
    _, run = _dense(sdpa, 1, 1, 1, 2048, 2048, 128, "top_left", -1, 5)
    assert run()[1] == 1
    # two query heads per key/value head, causal: 7 key tiles see 4 query
    # tiles on average, 8 pairs per unit (persistent); 8 key tiles, 9 pairs
    _, run = _dense(sdpa, 1, 4, 2, 896, 896, 128, "top_left", -1, 6)
    assert run()[1] == 2
    _, run = _dense(sdpa, 1, 4, 2, 1024, 1024, 128, "top_left", -1, 7)
    assert run()[1] == 1
    # forced either way
    _set(sdpa, 1)
    _, run = _dense(sdpa, 1, 2, 2, 1024, 1024, 64, "top_left", -1, 1)
    assert run()[1] == 1
    _set(sdpa, 2)
    _, run = _dense(sdpa, 1, 1, 1, 4096, 4096, 128, "none", -1, 2)
    assert run()[1] == 2
    _set(sdpa, 0)


def _packed_bwd(sdpa, lens_q, lens_kv, h, h_kv, d, seed):
    q, k, v, do, cu_q, cu_kv = sdpa_inputs.packed(lens_q, lens_kv, h, d, seed=seed, h_kv=h_kv)
    qc, kc, vc, doc, cq, ck = (x.cuda() for x in (q, k, v, do, cu_q, cu_kv))
    mq, mk = max(lens_q), max(lens_kv)
    o, lse = sdpa.attention_varlen(qc, kc, vc, cq, ck, mq, mk, scale=0.1, causal=True)
    got = sdpa.attention_varlen_bwd(qc, kc, vc, o, doc, lse, cq, ck, mq, mk, scale=0.1, causal=True)
    torch.cuda.synchronize()
    return (q, k, v, do, cu_q, cu_kv), got, sdpa.sdpa_last_backward_variant()


def test_packed_choice_by_sequence_count_and_length(sdpa):
    _set(sdpa, 0)
    lens = [40] * 128
    assert _packed_bwd(sdpa, lens, lens, 2, 2, 64, 3)[2] == 2
    many = [40] * 129
    assert _packed_bwd(sdpa, many, many, 2, 2, 64, 4)[2] == 1
    # long sequences (a mean of about 8 query tiles per key tile): one CTA per unit
    long = [2000, 1900, 2100, 2050]
    assert _packed_bwd(sdpa, long, long, 2, 2, 64, 5)[2] == 1
    _set(sdpa, 2)  # forced: long sequences run persistent, but the table holds 128 sequences
    assert _packed_bwd(sdpa, long, long, 2, 2, 64, 5)[2] == 2
    assert _packed_bwd(sdpa, many, many, 2, 2, 64, 4)[2] == 1
    _set(sdpa, 0)


DENSE = [
    # b, h, h_kv, s_q, s_kv, d, mask, window
    (2, 4, 4, 700, 700, 64, "top_left", -1),
    (1, 6, 2, 520, 900, 128, "bottom_right", -1),
    (2, 4, 1, 640, 640, 128, "top_left", 90),       # windows leave early key tiles unseen
    (1, 4, 4, 900, 300, 64, "bottom_right", 40),    # dead rows, unseen key tiles
    (3, 2, 2, 333, 333, 128, "none", -1),
]


@pytest.mark.parametrize("limit", [1, 5, 0], ids=["1cta", "5ctas", "per_sm"])
@pytest.mark.parametrize("case", DENSE, ids=lambda c: f"b{c[0]}h{c[1]}kv{c[2]}s{c[3]}x{c[4]}d{c[5]}_{c[6]}_w{c[7]}")
def test_persistent_dense_many_units_per_cta(sdpa, case, limit):
    b, h, h_kv, s_q, s_kv, d, mask, window = case
    (q, k, v, do, scale), run = _dense(sdpa, *case, seed=9000 + s_q + s_kv)
    _set(sdpa, 2, limit)
    got, used = run()
    assert used == 2
    _set(sdpa, 1)
    ref_gpu, used = run()
    assert used == 1
    _set(sdpa, 0)
    ref = oracle.sdpa_bwd_ex(q, k, v, do, scale, mask, window)
    for name, g, r, x in zip(("dq", "dk", "dv"), got, ref, ref_gpu):
        check_rel(g, r, GRAD_TOL, name)
        if name != "dq":
            assert torch.equal(g, x), f"{name}: persistent and per-tile kernels differ"
        else:
            check_rel(g, x.double().cpu().numpy(), 1e-2, "dq vs per-tile")


@pytest.mark.parametrize("limit", [2, 0], ids=["2ctas", "per_sm"])
def test_persistent_dense_deterministic(sdpa, limit):
    case = (1, 4, 2, 800, 800, 128, "top_left", -1)
    (q, k, v, do, scale), run = _dense(sdpa, *case, seed=9100, deterministic=True)
    _set(sdpa, 2, limit)
    a, used = run()
    b, _ = run()
    _set(sdpa, 0)
    assert used == 2
    for i in range(3):
        assert torch.equal(a[i], b[i])
    ref = oracle.sdpa_bwd_ex(q, k, v, do, scale, "top_left", -1)
    for name, g, r in zip(("dq", "dk", "dv"), a, ref):
        check_rel(g, r, GRAD_TOL, name)


@pytest.mark.parametrize("limit", [1, 7, 0], ids=["1cta", "7ctas", "per_sm"])
def test_persistent_packed_many_units_per_cta(sdpa, limit):
    """Sequences of every length class, some without queries or keys, two
    query heads per key/value head; 1 CTA walks the whole list."""
    g = np.random.default_rng(17)
    lens_q = g.integers(0, 700, 40).tolist()
    lens_kv = g.integers(0, 700, 40).tolist()
    lens_q[3] = 0
    lens_kv[8] = 0
    lens_q[11], lens_kv[11] = 1, 1
    _set(sdpa, 2, limit)
    (q, k, v, do, cu_q, cu_kv), got, used = _packed_bwd(sdpa, lens_q, lens_kv, 4, 2, 128, 18)
    _set(sdpa, 1)
    _, per_tile, _ = _packed_bwd(sdpa, lens_q, lens_kv, 4, 2, 128, 18)
    _set(sdpa, 0)
    assert used == 2
    ref = oracle.sdpa_varlen_bwd_ex(q, k, v, do, cu_q, cu_kv, 0.1, "top_left", -1)
    for name, x, r, y in zip(("dq", "dk", "dv"), got, ref, per_tile):
        check_rel(x, r, GRAD_TOL, name)
        if name != "dq":
            assert torch.equal(x, y), f"{name}: persistent and per-tile kernels differ"
